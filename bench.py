#!/usr/bin/env python
"""Benchmark of the Siddon projector pair: forward + matched backprojection.

One step = ctp_forward of the workload's phantom followed by ctp_backward of its
N(0,1) sinogram (the whole hot path: ray set-up, traversal-gather, zero-fill,
traversal-scatter).  Metric: giga ray-voxel segments per second, forward plus
backward, where one pass holds the float64 oracle's count of (ray, cell) pieces
longer than 1e-5 of the smallest cell width (tests/golden/segment_counts.json;
the plan's own counter agrees to 1e-6, tested).

    python bench.py [--gpus N] [--steps K] [--warmup W] [--config 1..5] [--impl reference]

With --gpus N > 1 (under torchrun) every rank runs an independent replica of the
workload; the line reports the units of all ranks over the slowest rank's time.
With --partition views the ranks share one workload instead: each projects its
contiguous shard of views, and the backward's partial volumes are summed with
one all-reduce (strong scaling).
"""

from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import tempfile
import sys
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import ctp_inputs as ci  # noqa: E402

METRIC = "Gray-segments/s (voxel-ray updates) fwd+bwd on 1 B300; % of BW roofline"
UNIT = "Gseg/s"
DEFAULT_CONFIG = 4
FALLBACK_HBM_GBS = 6400.0
CSRC = os.path.join(ROOT, "back_projection_ctp_b300", "csrc")
# ncu figures of profiled kernels (DRAM bytes per launch, limiting units), each
# with the hash of the kernel sources it was captured on
TRAFFIC_JSON = os.path.join(ROOT, "profiles", "traffic.json")
# calls per CUDA graph in the other workloads' per-call timings: enough that
# the microsecond-scale 2-D calls are not timed one launch at a time
PER_WORKLOAD_CALLS = 20


# ----------------------------------------------------------------- helpers
# Sources that compile into each profiled kernel (its code, its launch set-up
# and its parameter structs).
KERNEL_SOURCES = {
    "column_forward_kernel": ("ctp_column.cuh", "ctp_ray.cuh", "ctp_internal.h"),
    "column_backward_kernel": ("ctp_column.cuh", "ctp_ray.cuh", "ctp_internal.h"),
}


def source_hash(kernel: str) -> str:
    """Hash of a kernel's sources with comments and blank space removed, so that a
    stored ncu capture stays attached to unchanged code only."""
    import re
    h = hashlib.sha256()
    for name in KERNEL_SOURCES.get(kernel, sorted(os.listdir(CSRC))):
        with open(os.path.join(CSRC, name)) as fh:
            text = fh.read()
        text = re.sub(r"/\*.*?\*/", " ", text, flags=re.S)
        text = re.sub(r"//[^\n]*", " ", text)
        h.update(name.encode())
        h.update(" ".join(text.split()).encode())
    return h.hexdigest()[:16]


def golden_segments(idx: int) -> int:
    with open(os.path.join(ROOT, "tests", "golden", "segment_counts.json")) as fh:
        return int(json.load(fh)["full"][str(idx)]["segments"])


def hbm_peak():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as fh:
            peaks = json.load(fh)
        return float(peaks["hbm_gbs"]), "of measured"
    except (OSError, KeyError, ValueError):
        return FALLBACK_HBM_GBS, "of fallback"


# ------------------------------------------------------------ L2 bandwidth probes
def l2_peaks(dev, stream, repeats=5):
    """Measured L2 rates of this GPU (``libctp_probe.so``), best of ``repeats``:
    useful bytes/s of float reductions at full sector density (32 consecutive
    floats per warp instruction), 32-byte sectors/s of reductions at one float
    per sector, and bytes/s of coalesced loads that bypass L1; the buffers
    (64 MiB) stay in L2."""
    import ctypes
    import torch
    from back_projection_ctp_b300 import build as ctp_build
    lib = ctypes.CDLL(ctp_build.build_probe())
    lib.ctp_probe_l2_reduction.argtypes = [ctypes.c_void_p, ctypes.c_longlong, ctypes.c_int,
                                           ctypes.c_int, ctypes.c_void_p]
    lib.ctp_probe_l2_load.argtypes = [ctypes.c_void_p, ctypes.c_longlong, ctypes.c_int,
                                      ctypes.c_void_p, ctypes.c_void_p]
    lib.ctp_probe_sm_count.argtypes = [ctypes.POINTER(ctypes.c_int)]
    lib.ctp_probe_smem_accumulate.argtypes = [ctypes.c_int, ctypes.c_int, ctypes.c_void_p,
                                              ctypes.c_void_p]
    lib.ctp_probe_l2_bulk_reduction.argtypes = [ctypes.c_void_p, ctypes.c_longlong, ctypes.c_int,
                                                ctypes.c_int, ctypes.c_int, ctypes.c_void_p]
    sms = ctypes.c_int(0)
    if lib.ctp_probe_sm_count(ctypes.byref(sms)) != 0:
        raise RuntimeError("ctp_probe_sm_count failed")
    threads = sms.value * 8 * 256
    n = 16 << 20
    buf = torch.zeros(n, dtype=torch.float32, device=dev)
    sink = torch.zeros(1, dtype=torch.float32, device=dev)
    sp = stream.cuda_stream

    def best(launch, units):
        launch()
        torch.cuda.synchronize(dev)
        times = []
        for _ in range(repeats):
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record(stream)
            launch()
            b.record(stream)
            torch.cuda.synchronize(dev)
            times.append(a.elapsed_time(b) * 1e-3)
        return units / min(times)

    def check(st):
        if st != 0:
            raise RuntimeError(f"L2 probe failed ({st})")

    it_red, it_load = 16000, 4000
    red = best(lambda: check(lib.ctp_probe_l2_reduction(buf.data_ptr(), n, it_red, 0, sp)),
               4.0 * threads * it_red)
    sectors = best(lambda: check(lib.ctp_probe_l2_reduction(buf.data_ptr(), n, it_load, 1, sp)),
                   1.0 * threads * it_load)
    load = best(lambda: check(lib.ctp_probe_l2_load(buf.data_ptr(), n, it_load, sink.data_ptr(),
                                                    sp)), 16.0 * threads * it_load)
    # shared-memory float accumulation (adds per clock per SM at the maximum clock)
    smem = {}
    for mode, name in ((0, "atomic_distinct_words"), (1, "load_add_store"),
                       (2, "atomic_4_lanes_per_word")):
        rate = best(lambda: check(lib.ctp_probe_smem_accumulate(it_load, mode, sink.data_ptr(),
                                                                sp)), 1.0 * threads * it_load)
        smem[name] = rate / sms.value / 2.032e9
    # bulk reductions of the async copy engine: 256-byte runs from shared memory,
    # 8 issuing lanes per warp (full sectors, like a dense reduction stream)
    it_bulk, run, lanes = 200, 256, 8
    bulk = best(lambda: check(lib.ctp_probe_l2_bulk_reduction(buf.data_ptr(), n, it_bulk, run,
                                                              lanes, sp)),
                1.0 * run * (threads // 32) * lanes * it_bulk)
    return {"reduction_gbs": red / 1e9, "reduction_sectors_per_s": sectors,
            "load_gbs": load / 1e9, "bulk_reduction_gbs": bulk / 1e9,
            "smem_adds_per_clock_per_sm": smem,
            "how": "libctp_probe.so: 8 blocks x 256 threads per SM over a 64 MiB buffer held "
                   "in L2 (shared memory: 256 words per block); best of 5 launches timed "
                   "with CUDA events"}


def stored_traffic(kernel: str, workload: str):
    """DRAM bytes per launch from the committed ncu summary, if it was taken on
    the current kernel sources; else None."""
    path = TRAFFIC_JSON
    try:
        with open(path) as fh:
            rec = json.load(fh)
    except (OSError, ValueError):
        return None
    entry = rec.get(kernel, {}).get(workload)
    if not entry or entry.get("source_hash") != source_hash(kernel):
        return None
    return entry.get("dram_bytes_per_launch")


def geometry_of(w, frames):
    from back_projection_ctp_b300 import Geometry
    return Geometry(ndim=w.ndim, beam=w.beam, src=frames["src"], det_centre=frames["det_centre"],
                    det_u=frames["det_u"], det_v=frames["det_v"], n_u=w.n_u, n_v=w.n_v,
                    pitch_u=w.pitch_u, pitch_v=w.pitch_v, offset_u=w.offset_u,
                    offset_v=w.offset_v)


def volume_of(w):
    from back_projection_ctp_b300 import Volume
    return Volume(shape=w.shape, spacing=w.spacing, origin=w.origin)


class ClockSampler:
    """nvidia-smi clocks and throttle reasons sampled every 200 ms, logged to
    $CTP_BENCH_LOG_DIR (default: a temporary directory) as clocks_rank<i>.csv."""

    QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None
        log_dir = os.environ.get("CTP_BENCH_LOG_DIR") or tempfile.gettempdir()
        self.path = os.path.join(log_dir, f"clocks_rank{index}.csv")

    def start(self):
        try:
            os.makedirs(os.path.dirname(self.path), exist_ok=True)
            self.fh = open(self.path, "w")
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.index}", f"--query-gpu={self.QUERY}",
                 "--format=csv,noheader,nounits", "-lms", "200"],
                stdout=self.fh, stderr=subprocess.DEVNULL)
        except OSError:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.fh.close()
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        with open(self.path) as fh:
            for line in fh:
                parts = [p.strip() for p in line.split(",")]
                if len(parts) < 9:
                    continue
                try:
                    sm.append(float(parts[1]))
                    smax.append(float(parts[2]))
                except ValueError:
                    continue
                for name, val in zip(names, parts[5:9]):
                    if val.lower() == "active":
                        reasons.add(name)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"]}
        loaded = [s for s in sm if s > 0.5 * max(sm)] or sm
        return {"sm_mhz": statistics.median(loaded), "sm_max_mhz": max(smax),
                "reasons": sorted(reasons), "samples": len(sm)}


# ------------------------------------------------------------ distributed
def dist_setup(n_gpus: int):
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch
        import torch.distributed as dist
        backend = "nccl" if torch.cuda.is_available() else "gloo"
        if backend == "nccl":
            torch.cuda.set_device(local)
        dist.init_process_group(backend)
    return world, rank, local


def barrier(world: int):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(value: float, world: int) -> float:
    if world <= 1:
        return value
    import torch
    import torch.distributed as dist
    dev = "cuda" if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([value], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


# ----------------------------------------------------------------- oracle arm
def oracle_sample_rate(w, vol, y, budget_s: float = 15.0):
    """The float64 oracle, as it stands, on a bounded sample of the workload:
    forward and backward over the rays of the first m views, m sized so the
    timed work is about budget_s seconds.  Returns (Gseg/s of forward +
    backward, sample text, cores, seconds, {forward / backward Gseg/s})."""
    import oracle
    scan = oracle.Scan.from_workload(w, ci.frames(w))
    cores = len(os.sched_getaffinity(0)) if hasattr(os, "sched_getaffinity") else os.cpu_count()
    per_view = w.n_u * w.n_v
    # probe one view (untimed for the result) to size the sample
    t = time.perf_counter()
    oracle.forward(scan, vol, 0, per_view, threads=cores)
    oracle.backward(scan, y[:per_view], 0, per_view, threads=cores)
    probe = time.perf_counter() - t
    m = int(max(1, min(w.n_views, budget_s // max(probe, 1e-3))))
    ray1 = m * per_view
    segs = oracle.segment_count(scan, 0, ray1, threads=cores)
    t = time.perf_counter()
    oracle.forward(scan, vol, 0, ray1, threads=cores)
    t_fwd = time.perf_counter() - t
    t = time.perf_counter()
    oracle.backward(scan, y[:ray1], 0, ray1, threads=cores)
    t_bwd = time.perf_counter() - t
    dt = t_fwd + t_bwd
    sample = (f"views 0..{m - 1} of {w.n_views} ({ray1} rays, {segs} segments), forward + "
              f"backward, float64 C oracle, {cores} threads, {dt:.1f} s")
    parts = {"forward_gseg_per_s": segs / t_fwd / 1e9, "backward_gseg_per_s": segs / t_bwd / 1e9}
    return 2.0 * segs / dt / 1e9, sample, cores, dt, parts


def run_reference(args, w, world, rank):
    if rank != 0:
        return 0
    vol = ci.phantom(w)
    y = ci.sinogram_noise(w).ravel()
    rates, samples = [], []
    for step in range(args.warmup + args.steps):
        rate, sample, cores, dt, parts = oracle_sample_rate(w, vol, y, budget_s=args.ref_budget)
        if step >= args.warmup:
            rates.append(rate)
            samples.append(dt)
    value = statistics.median(rates)
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": 1000 * statistics.median(samples), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": w.name, "note": "each step is a bounded sample of the workload"},
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": cores, "kind": "oracle",
                         "sample": sample, **parts},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return 0


# ------------------------------------------------------------------ GPU arm
def time_pair(ctp, plan, d_vol, d_y, d_sino, d_g, steps, warmup, dev, stream, calls=None):
    """Device times (ms) of one forward call and one backward call on the
    caller's stream, each the median over three replays (after an untimed one)
    of a CUDA graph of ``calls`` calls (default ``steps``) between CUDA events;
    plus the graph of ``steps`` forward + backward steps and the timing function
    for the caller's timed region."""
    import torch

    for _ in range(warmup):
        ctp.ctp_forward(plan, d_vol, d_sino, stream)
        ctp.ctp_backward(plan, d_y, d_g, stream)
    torch.cuda.synchronize(dev)

    # The calls only enqueue kernels and a memset, so they capture as they are.
    def capture(body, n):
        graph = torch.cuda.CUDAGraph()
        side = torch.cuda.Stream(dev)
        side.wait_stream(torch.cuda.current_stream(dev))
        with torch.cuda.stream(side), torch.cuda.graph(graph, stream=side):
            cur = torch.cuda.current_stream(dev)
            for _ in range(n):
                body(cur)
        torch.cuda.synchronize(dev)
        return graph

    calls = calls or steps
    g_steps = capture(lambda st: (ctp.ctp_forward(plan, d_vol, d_sino, st),
                                  ctp.ctp_backward(plan, d_y, d_g, st)), steps)
    g_fwd = capture(lambda st: ctp.ctp_forward(plan, d_vol, d_sino, st), calls)
    g_bwd = capture(lambda st: ctp.ctp_backward(plan, d_y, d_g, st), calls)
    for graph in (g_steps, g_fwd, g_bwd):  # one untimed replay each (graph upload)
        graph.replay()
    torch.cuda.synchronize(dev)

    def timed(graph):
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        graph.replay()
        b.record(stream)
        torch.cuda.synchronize(dev)
        return a.elapsed_time(b)

    def per_call(graph):
        return statistics.median(timed(graph) for _ in range(3)) / calls

    return timed, g_steps, per_call(g_fwd), per_call(g_bwd)


def kernel_of(path, call):
    return {"column": {"forward": "column_forward_kernel", "backward": "column_backward_kernel"},
            "plane": {"forward": "plane_forward_kernel", "backward": "plane_backward_kernel"},
            "ray": {"forward": "ray_forward_kernel", "backward": "ray_backward_kernel"}}[path][call]


# ncu figures of the committed summaries (profiles/): the unit that limits each
# dominant kernel, by kernel and workload
def stored_ncu(kernel: str, workload: str):
    path = TRAFFIC_JSON
    try:
        with open(path) as fh:
            rec = json.load(fh)
    except (OSError, ValueError):
        return None
    entry = rec.get(kernel, {}).get(workload)
    if not entry or entry.get("source_hash") != source_hash(kernel):
        return None
    return entry.get("ncu")


def per_workload(args, ctp, dev, stream, peaks, skip):
    """Forward and backward device times of every workload but ``skip`` (the
    headline one), with the same graphs and the same units; each workload's
    phantom and N(0,1) sinogram as in the parity tests."""
    import torch
    out = {}
    hbm, _ = hbm_peak()
    for idx in sorted(ci.WORKLOADS):
        if idx == skip:
            continue
        w = ci.get(idx)
        plan = ctp.ctp_plan(geometry_of(w, ci.frames(w)), volume_of(w), args.path)
        d_vol = torch.from_numpy(ci.phantom(w)).to(dev)
        d_y = torch.from_numpy(ci.sinogram_noise(w)).to(dev)
        d_sino = torch.empty(plan.sino_shape, dtype=torch.float32, device=dev)
        d_g = torch.empty(plan.vol_shape, dtype=torch.float32, device=dev)
        timed, g_steps, fwd_ms, bwd_ms = time_pair(ctp, plan, d_vol, d_y, d_sino, d_g,
                                                   args.steps, args.warmup, dev, stream,
                                                   calls=max(args.steps, PER_WORKLOAD_CALLS))
        step_ms = timed(g_steps) / args.steps
        seg = golden_segments(idx)
        out[w.name] = {
            "path": plan.path, "segments_per_pass": seg, "fwd_ms": fwd_ms, "bwd_ms": bwd_ms,
            "ms_per_step": step_ms, "gseg_per_s": 2.0 * seg / (step_ms * 1e-3) / 1e9,
            "fwd_frac_l2_load": 4.0 * seg / (fwd_ms * 1e-3) / 1e9 / peaks["load_gbs"],
            "bwd_frac_l2_reduction": 4.0 * seg / (bwd_ms * 1e-3) / 1e9 / peaks["reduction_gbs"],
            "fwd_frac_hbm_equivalent": 4.0 * seg / (fwd_ms * 1e-3) / 1e9 / hbm,
            "bwd_frac_hbm_equivalent": 4.0 * seg / (bwd_ms * 1e-3) / 1e9 / hbm,
        }
        del g_steps
        plan.destroy()
        del d_vol, d_y, d_sino, d_g
        torch.cuda.empty_cache()
    return out


def run_gpu(args, w, world, rank, local):
    """Time K steps of forward + backward on this rank's GPU."""
    import torch
    import back_projection_ctp_b300 as ctp

    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    frames = ci.frames(w)
    vol_h = ci.phantom(w)
    y_h = ci.sinogram_noise(w)
    plan = ctp.ctp_plan(geometry_of(w, frames), volume_of(w), args.path, options=args.plan_options)
    if args.views is None:
        segments = golden_segments(args.config)
        seg_source = "float64 oracle (tests/golden/segment_counts.json)"
    else:
        segments = ctp.ctp_segment_count(plan)
        seg_source = "plan counter (reduced-view scan)"

    stream = torch.cuda.current_stream(dev)
    d_vol = torch.from_numpy(vol_h).to(dev)
    d_y = torch.from_numpy(y_h).to(dev)
    d_sino = torch.empty(plan.sino_shape, dtype=torch.float32, device=dev)
    d_g = torch.empty(plan.vol_shape, dtype=torch.float32, device=dev)

    timed, g_steps, fwd_ms, bwd_ms = time_pair(ctp, plan, d_vol, d_y, d_sino, d_g, args.steps,
                                               args.warmup, dev, stream)
    sampler = ClockSampler(local)
    sampler.start()
    time.sleep(0.3)
    barrier(world)
    torch.cuda.synchronize(dev)
    total_ms = timed(g_steps)
    torch.cuda.synchronize(dev)
    barrier(world)
    clocks = sampler.stop()
    total_ms = max_over_ranks(total_ms, world)
    ms_per_step = total_ms / args.steps
    value = world * 2.0 * segments / (ms_per_step * 1e-3) / 1e9

    # end to end through the host-buffer C-ABI calls (pinned host memory)
    vol_pin = torch.from_numpy(vol_h).pin_memory().numpy()
    y_pin = torch.from_numpy(y_h).pin_memory().numpy()
    sino_pin = torch.empty(plan.sino_shape, dtype=torch.float32).pin_memory().numpy()
    g_pin = torch.empty(plan.vol_shape, dtype=torch.float32).pin_memory().numpy()
    ctp.ctp_forward_host(plan, vol_pin, sino_pin, stream)
    ctp.ctp_backward_host(plan, y_pin, g_pin, stream)
    e2e_steps = max(1, min(args.steps, 3))
    barrier(world)
    torch.cuda.synchronize(dev)
    t0 = time.perf_counter()
    for _ in range(e2e_steps):
        ctp.ctp_forward_host(plan, vol_pin, sino_pin, stream)
        ctp.ctp_backward_host(plan, y_pin, g_pin, stream)
    torch.cuda.synchronize(dev)
    e2e_s = max_over_ranks((time.perf_counter() - t0) / e2e_steps, world)
    barrier(world)
    e2e_value = world * 2.0 * segments / e2e_s / 1e9
    bytes_io = 4 * (w.n_voxels + w.n_rays)

    # Roofline of the dominant call.  Its segment stream (4 algorithmic bytes
    # per segment: one voxel read per forward piece, one float reduction per
    # backward piece) is served by L1 / L2, so the bound is L2: the backward
    # against the measured rate at which L2 takes float reductions at full
    # sector density, the forward against L2's load rate.  The same bytes over
    # the measured HBM copy bandwidth (an HBM-equivalent fraction) and the ncu
    # DRAM traffic over it (the measured DRAM fraction) are reported beside it.
    del g_steps
    peaks = l2_peaks(dev, stream)
    dominant = "backward" if bwd_ms >= fwd_ms else "forward"
    dom_ms = max(bwd_ms, fwd_ms)
    achieved = 4.0 * segments / (dom_ms * 1e-3) / 1e9
    l2_peak = peaks["reduction_gbs"] if dominant == "backward" else peaks["load_gbs"]
    hbm, hbm_src = hbm_peak()
    kernel_name = kernel_of(plan.path, dominant)
    traffic = stored_traffic(kernel_name, w.name)
    # kernels of this library per step: column / plane = layout pass + walk, twice
    launches_per_step = 2 if plan.path == "ray" else 4
    plan_path = plan.path
    plan.destroy()
    del d_vol, d_y, d_sino, d_g
    torch.cuda.empty_cache()
    others = per_workload(args, ctp, dev, stream, peaks, args.config) \
        if (world == 1 and args.views is None and not args.no_per_workload) else None

    if rank == 0:
        cpu = None
        if world == 1 and not args.no_cpu_baseline:
            rate, sample, cores, _, parts = oracle_sample_rate(w, vol_h, y_h.ravel(),
                                                               args.ref_budget)
            cpu = {"value": rate, "unit": UNIT, "cores": cores, "kind": "oracle", "sample": sample,
                   **parts}
        line = {
            "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": ms_per_step, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f32", "data": "synthetic",
            "config": {"workload": w.name, "shape_DHW": list(w.shape),
                       "spacing_DHW": list(w.spacing), "views": w.n_views,
                       "detector_vu": [w.n_v, w.n_u], "segments_per_pass": segments,
                       "segments_from": seg_source,
                       "path": plan_path, "parallelism": f"replicas{world}",
                       "l2": "inputs larger than L2 (no flush)" if 4 * w.n_voxels > 126e6
                       else "inputs smaller than L2 (no flush)",
                       "fwd_ms": fwd_ms, "bwd_ms": bwd_ms,
                       "per_workload": others},
            "roofline": {
                "bound": "l2", "achieved": achieved, "peak": l2_peak, "unit": "GB/s",
                "frac": achieved / l2_peak, "traffic": traffic, "kernel": kernel_name,
                "call": dominant,
                "peak_source": ("measured in this run: L2 float reductions at full sector "
                                "density" if dominant == "backward" else
                                "measured in this run: L2 loads bypassing L1"),
                "l2_probe": peaks,
                "hbm_equivalent": {"peak": hbm, "frac": achieved / hbm,
                                   "note": f"the same 4 B per segment over the HBM copy "
                                           f"bandwidth ({hbm_src}); not a DRAM measurement"},
                "dram_frac": (traffic / (dom_ms * 1e-3) / 1e9 / hbm) if traffic else None,
                # the floor of any implementation's DRAM traffic for one call:
                # its input and output arrays once each
                "compulsory_bytes": 4 * (w.n_voxels + w.n_rays),
                "ncu": stored_ncu(kernel_name, w.name),
                "note": f"4 algorithmic bytes per segment over the {dominant} call's event "
                        "time; dram_frac = the ncu DRAM bytes of one launch over the same "
                        "time and the HBM copy bandwidth"},
            "cpu_baseline": cpu,
            "e2e": {"value": e2e_value, "unit": UNIT, "h2d_bytes_per_step": bytes_io,
                    "d2h_bytes_per_step": bytes_io, "ms_per_step": e2e_s * 1e3},
            "gpu_launches": launches_per_step * args.steps,
            "timing": "one CUDA graph of K steps replayed between CUDA events on the calls' stream",
            "clocks": clocks,
        }
        print(json.dumps(line), flush=True)
    return 0


# ------------------------------------------------- view-partitioned (strong scaling)
def run_partitioned(args, w, world, rank, local):
    """One workload sharded by views over the ranks (one GPU each): each rank
    projects its views and backprojects them into a full-volume partial, and
    one all-reduce (sum) of the volume per backward gives A^T y on every rank.
    Total work is fixed as ranks are added ("strong" scaling)."""
    import torch
    import back_projection_ctp_b300 as ctp

    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    stream = torch.cuda.current_stream(dev)
    frames = ci.frames(w)
    proj = ctp.ViewShardedProjector(geometry_of(w, frames), volume_of(w), args.path)
    segments = golden_segments(args.config) if args.views is None else None
    vol_h = ci.phantom(w)
    y_h = np.ascontiguousarray(ci.sinogram_noise(w)[proj.v0:proj.v1])
    d_vol = torch.from_numpy(vol_h).to(dev)
    d_y = torch.from_numpy(y_h).to(dev)
    d_sino = torch.empty(proj.local_sino_shape, dtype=torch.float32, device=dev)
    d_g = torch.empty(w.shape, dtype=torch.float32, device=dev)
    if segments is None:
        counts = torch.tensor([float(ctp.ctp_segment_count(proj.op.plan))], dtype=torch.float64,
                              device=dev)
        proj.all_reduce(counts)
        segments = int(counts.item())

    def step():
        proj.forward(d_vol, d_sino)
        proj.backward(d_y, d_g)

    def timed(body, n):
        barrier(world)
        torch.cuda.synchronize(dev)
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        for _ in range(n):
            body()
        b.record(stream)
        torch.cuda.synchronize(dev)
        barrier(world)
        return a.elapsed_time(b)

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize(dev)
    sampler = ClockSampler(local)
    sampler.start()
    time.sleep(0.3)
    total_ms = max_over_ranks(timed(step, args.steps), world)
    clocks = sampler.stop()
    ms_per_step = total_ms / args.steps
    value = 2.0 * segments / (ms_per_step * 1e-3) / 1e9
    fwd_ms = max_over_ranks(timed(lambda: proj.forward(d_vol, d_sino), args.steps), world) / args.steps
    bwd_ms = max_over_ranks(timed(lambda: proj.backward(d_y, d_g), args.steps), world) / args.steps

    # end to end: every step each rank uploads the volume and its sinogram rows
    # from pinned memory, runs the pair (with the all-reduce) and downloads its
    # sinogram rows and the volume
    vol_pin = torch.from_numpy(vol_h).pin_memory()
    y_pin = torch.from_numpy(y_h).pin_memory()
    sino_pin = torch.empty(proj.local_sino_shape, dtype=torch.float32).pin_memory()
    g_pin = torch.empty(w.shape, dtype=torch.float32).pin_memory()

    def e2e_step():
        d_vol.copy_(vol_pin, non_blocking=True)
        proj.forward(d_vol, d_sino)
        sino_pin.copy_(d_sino, non_blocking=True)
        d_y.copy_(y_pin, non_blocking=True)
        proj.backward(d_y, d_g)
        g_pin.copy_(d_g, non_blocking=True)
        torch.cuda.synchronize(dev)

    e2e_step()
    e2e_steps = max(1, min(args.steps, 3))
    barrier(world)
    t0 = time.perf_counter()
    for _ in range(e2e_steps):
        e2e_step()
    e2e_s = max_over_ranks((time.perf_counter() - t0) / e2e_steps, world)
    e2e_value = 2.0 * segments / e2e_s / 1e9
    io = 4 * (world * w.n_voxels + w.n_rays)
    plan_path = proj.op.plan.path
    if rank == 0:
        line = {
            "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms_per_step,
            "higher_is_better": True, "scaling": "strong", "vs_baseline": None, "dtype": "f32",
            "data": "synthetic",
            "config": {"workload": w.name, "views": w.n_views, "detector_vu": [w.n_v, w.n_u],
                       "segments_per_pass": segments, "path": plan_path,
                       "parallelism": f"views{world}",
                       "views_per_rank": [list(ctp.view_shard(w.n_views, world, r))
                                          for r in range(world)],
                       "collective": "one all-reduce (sum) of the volume per backward",
                       "fwd_ms": fwd_ms, "bwd_ms_with_all_reduce": bwd_ms,
                       "l2": "inputs larger than L2 (no flush)" if 4 * w.n_voxels > 126e6
                       else "inputs smaller than L2 (no flush)"},
            "e2e": {"value": e2e_value, "unit": UNIT, "h2d_bytes_per_step": io,
                    "d2h_bytes_per_step": io, "ms_per_step": e2e_s * 1e3},
            "gpu_launches": (2 if plan_path == "ray" else 4) * args.steps * world,
            "timing": "K eager steps between CUDA events on the calls' stream, max over ranks",
            "clocks": clocks,
        }
        print(json.dumps(line), flush=True)
    proj.destroy()
    return 0


# ------------------------------------------------------ analytical FDK (second op)
FDK_METRIC = "FDK voxel-view updates/s (ramp filter + weighted gather) on 1 B300"
FDK_UNIT = "Gvox-view/s"
# FP32 lanes x 2 flops x clock: 148 SMs x 128 lanes x 2 x 2.032 GHz (no tensor cores)
FP32_PEAK_TFLOPS = 148 * 128 * 2 * 2.032e9 / 1e12
# algorithmic float32 flops of one voxel-view update: three linear interpolations
# (a subtract and a multiply-add each: 3 flops) and the weighted accumulate (a
# multiply-add: 2 flops)
FDK_FLOPS_PER_UPDATE = 11


def oracle_fdk_rate(w, p, budget_s):
    """The float64 FDK oracle on a bounded sample: the first m views, filtered and
    gathered over the central z slice.  Returns (Gvox-view/s, sample text, cores)."""
    import oracle
    from oracle import fdk as ofdk
    cores = len(os.sched_getaffinity(0)) if hasattr(os, "sched_getaffinity") else os.cpu_count()
    scan = oracle.Scan.from_workload(w, ci.frames(w))
    D, H, W = w.shape
    kc = D // 2
    vox = np.stack(np.meshgrid([kc], np.arange(H), np.arange(W), indexing="ij"), -1).reshape(-1, 3)
    vw = np.full(w.n_views, np.pi / w.n_views)

    def run(m):
        sub = oracle.Scan(w.beam, *(a[:m] for a in scan.arrays), w.n_u, w.n_v, w.pitch_u,
                          w.pitch_v, w.shape, w.spacing, w.origin, w.offset_u, w.offset_v, w.ndim)
        t = time.perf_counter()
        q = ofdk.filter_sinogram(sub, p[:m], vw[:m])
        ofdk.weighted_backproject(sub, q, voxels=vox)
        return time.perf_counter() - t

    probe = run(1)
    m = int(max(1, min(w.n_views, budget_s // max(probe, 1e-3))))
    dt = run(m)
    sample = (f"views 0..{m - 1} of {w.n_views}: ramp filter of those views and weighted gather "
              f"over the central z slice ({H * W} voxels), float64 numpy oracle, {dt:.1f} s")
    return H * W * m / dt / 1e9, sample, cores


def run_fdk(args, w, world, rank, local):
    """Time K FDK reconstructions (ramp filter + weighted gather) of the workload."""
    import torch
    import back_projection_ctp_b300 as ctp

    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    frames = ci.frames(w)
    p_h = ci.sinogram_noise(w).reshape(w.n_views, w.n_v, w.n_u)
    plan = ctp.ctp_plan(geometry_of(w, frames), volume_of(w), args.path)
    stream = torch.cuda.current_stream(dev)
    d_p = torch.from_numpy(p_h).to(dev)
    d_q = torch.empty_like(d_p)
    d_vol = torch.empty(plan.vol_shape, dtype=torch.float32, device=dev)
    d_vw = torch.from_numpy(ctp.full_scan_view_weights(w.n_views)).to(dev)
    for _ in range(args.warmup):
        ctp.ctp_fdk(plan, d_p, d_q, d_vol, d_vw, "ramlak", stream)
    torch.cuda.synchronize(dev)

    def capture(body):
        graph = torch.cuda.CUDAGraph()
        side = torch.cuda.Stream(dev)
        side.wait_stream(torch.cuda.current_stream(dev))
        with torch.cuda.stream(side), torch.cuda.graph(graph, stream=side):
            cur = torch.cuda.current_stream(dev)
            for _ in range(args.steps):
                body(cur)
        torch.cuda.synchronize(dev)
        return graph

    g_steps = capture(lambda st: ctp.ctp_fdk(plan, d_p, d_q, d_vol, d_vw, "ramlak", st))
    g_filter = capture(lambda st: ctp.ctp_ramp_filter(plan, d_p, d_q, d_vw, "ramlak", False, st))
    g_gather = capture(lambda st: ctp.ctp_weighted_backproject(plan, d_q, d_vol, st))
    d_t = torch.empty_like(d_p)
    g_transpose = capture(lambda st: ctp.ctp_weighted_backproject_transpose(plan, d_vol, d_t, st))
    g_steps.replay()
    torch.cuda.synchronize(dev)

    def timed(graph):
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        graph.replay()
        b.record(stream)
        torch.cuda.synchronize(dev)
        return a.elapsed_time(b)

    sampler = ClockSampler(local)
    sampler.start()
    time.sleep(0.3)
    barrier(world)
    torch.cuda.synchronize(dev)
    total_ms = timed(g_steps)
    torch.cuda.synchronize(dev)
    barrier(world)
    clocks = sampler.stop()
    total_ms = max_over_ranks(total_ms, world)
    filter_ms = timed(g_filter) / args.steps
    gather_ms = timed(g_gather) / args.steps
    transpose_ms = timed(g_transpose) / args.steps
    ms_per_step = total_ms / args.steps
    updates = w.n_voxels * w.n_views
    value = world * updates / (ms_per_step * 1e-3) / 1e9

    # end to end: pinned sinogram up, FDK, volume down, every step
    p_pin = torch.from_numpy(p_h).pin_memory()
    v_pin = torch.empty(plan.vol_shape, dtype=torch.float32).pin_memory()
    e2e_steps = max(1, min(args.steps, 3))
    for it in range(e2e_steps + 1):
        if it == 1:
            torch.cuda.synchronize(dev)
            t0 = time.perf_counter()
        d_p.copy_(p_pin, non_blocking=True)
        ctp.ctp_fdk(plan, d_p, d_q, d_vol, d_vw, "ramlak", stream)
        v_pin.copy_(d_vol, non_blocking=True)
        torch.cuda.synchronize(dev)
    e2e_s = max_over_ranks((time.perf_counter() - t0) / e2e_steps, world)
    e2e_value = world * updates / e2e_s / 1e9

    achieved = FDK_FLOPS_PER_UPDATE * updates / (gather_ms * 1e-3) / 1e12
    if rank == 0:
        cpu = None
        if world == 1 and not args.no_cpu_baseline:
            rate, sample, cores = oracle_fdk_rate(w, p_h, args.ref_budget)
            cpu = {"value": rate, "unit": FDK_UNIT, "cores": cores, "kind": "oracle",
                   "sample": sample}
        line = {
            "metric": FDK_METRIC, "value": value, "unit": FDK_UNIT, "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms_per_step,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f32",
            "data": "synthetic",
            "config": {"workload": w.name, "op": "fdk", "shape_DHW": list(w.shape),
                       "views": w.n_views, "detector_vu": [w.n_v, w.n_u], "ramp": "ramlak",
                       "parallelism": f"replicas{world}",
                       "l2": "inputs larger than L2 (no flush)" if 4 * w.n_rays > 126e6
                       else "inputs smaller than L2 (no flush)",
                       "filter_ms": filter_ms, "gather_ms": gather_ms,
                       "gather_transpose_ms": transpose_ms},
            "roofline": {"bound": "alu", "achieved": achieved, "peak": FP32_PEAK_TFLOPS,
                         "unit": "TFLOP/s", "frac": achieved / FP32_PEAK_TFLOPS, "traffic": None,
                         "kernel": "wbp_gather_kernel", "call": "gather",
                         "note": f"{FDK_FLOPS_PER_UPDATE} float32 flops per voxel-view update "
                                 "over the gather's event time; peak = 148 SMs x 128 lanes x 2 "
                                 "x 2.032 GHz (derived from unit counts and clock)"},
            "cpu_baseline": cpu,
            "e2e": {"value": e2e_value, "unit": FDK_UNIT, "h2d_bytes_per_step": 4 * w.n_rays,
                    "d2h_bytes_per_step": 4 * w.n_voxels, "ms_per_step": e2e_s * 1e3},
            "gpu_launches": 2 * args.steps,
            "timing": "one CUDA graph of K steps replayed between CUDA events on the calls' stream",
            "clocks": clocks,
        }
        print(json.dumps(line), flush=True)
    plan.destroy()
    return 0


# ------------------------------------------------ geometry gradients (third op)
GEOM_METRIC = "Geometry-gradient Gseg/s (ray walk with crossing terms) on 1 B300"


def run_geometry(args, w, world, rank, local):
    """Time K geometry vector-Jacobian products (all views) of the workload."""
    import torch
    import back_projection_ctp_b300 as ctp

    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    frames = ci.frames(w)
    plan = ctp.ctp_plan(geometry_of(w, frames), volume_of(w), args.path,
                        options=args.plan_options)
    segments = golden_segments(args.config) if args.views is None else ctp.ctp_segment_count(plan)
    stream = torch.cuda.current_stream(dev)
    d_vol = torch.from_numpy(ci.phantom(w)).to(dev)
    d_y = torch.from_numpy(ci.sinogram_noise(w).reshape(plan.sino_shape)).to(dev)
    grad = torch.empty((w.n_views, 4, 3), dtype=torch.float64, device=dev)
    for _ in range(args.warmup):
        ctp.ctp_geometry_vjp(plan, d_vol, d_y, grad, stream)
    torch.cuda.synchronize(dev)
    graph = torch.cuda.CUDAGraph()
    side = torch.cuda.Stream(dev)
    side.wait_stream(torch.cuda.current_stream(dev))
    with torch.cuda.stream(side), torch.cuda.graph(graph, stream=side):
        cur = torch.cuda.current_stream(dev)
        for _ in range(args.steps):
            ctp.ctp_geometry_vjp(plan, d_vol, d_y, grad, cur)
    torch.cuda.synchronize(dev)
    graph.replay()
    torch.cuda.synchronize(dev)
    sampler = ClockSampler(local)
    sampler.start()
    time.sleep(0.3)
    barrier(world)
    torch.cuda.synchronize(dev)
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a.record(stream)
    graph.replay()
    b.record(stream)
    torch.cuda.synchronize(dev)
    barrier(world)
    clocks = sampler.stop()
    ms = max_over_ranks(a.elapsed_time(b), world) / args.steps
    value = world * segments / (ms * 1e-3) / 1e9
    achieved = 4.0 * segments / (ms * 1e-3) / 1e9
    peak, peak_src = hbm_peak()
    if rank == 0:
        cpu = None
        if world == 1 and not args.no_cpu_baseline:
            import oracle
            scan = oracle.Scan.from_workload(w, frames)
            cores = len(os.sched_getaffinity(0))
            per = w.n_u * w.n_v
            t = time.perf_counter()
            oracle.geometry_vjp(_first_views(oracle, scan, w, 1), ci.phantom(w),
                                np.ones(per, np.float32), threads=cores)
            probe = time.perf_counter() - t
            m = int(max(1, min(w.n_views, args.ref_budget // max(probe, 1e-3))))
            sub = _first_views(oracle, scan, w, m)
            segs = oracle.segment_count(sub, threads=cores)
            t = time.perf_counter()
            oracle.geometry_vjp(sub, ci.phantom(w), np.ones(m * per, np.float32), threads=cores)
            dt = time.perf_counter() - t
            cpu = {"value": segs / dt / 1e9, "unit": UNIT, "cores": cores, "kind": "oracle",
                   "sample": f"views 0..{m - 1} of {w.n_views}: float64 C oracle geometry "
                             f"gradient, {segs} segments, {dt:.1f} s"}
        line = {
            "metric": GEOM_METRIC, "value": value, "unit": UNIT, "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f32",
            "data": "synthetic",
            "config": {"workload": w.name, "op": "geometry", "views": w.n_views,
                       "detector_vu": [w.n_v, w.n_u], "segments_per_pass": segments,
                       "parallelism": f"replicas{world}"},
            "roofline": {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s",
                         "frac": achieved / peak, "traffic": None,
                         "kernel": "geometry_vjp_kernel", "call": "geometry_vjp",
                         "note": f"4 B per segment over the call's event time; peak {peak_src}"},
            "cpu_baseline": cpu,
            "gpu_launches": args.steps,
            "timing": "one CUDA graph of K calls replayed between CUDA events on the calls' stream",
            "clocks": clocks,
        }
        print(json.dumps(line), flush=True)
    plan.destroy()
    return 0


def _first_views(oracle, scan, w, m):
    return oracle.Scan(w.beam, *(a[:m] for a in scan.arrays), w.n_u, w.n_v, w.pitch_u,
                       w.pitch_v, w.shape, w.spacing, w.origin, w.offset_u, w.offset_v, w.ndim)


def main(argv=None):
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=10)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--config", type=int, default=DEFAULT_CONFIG)
    ap.add_argument("--views", type=int, default=None,
                    help="replace the workload's number of views (same arc); for profiling "
                         "captures of the same kernels on a shorter scan")
    ap.add_argument("--impl", default="ctp", choices=["ctp", "reference"])
    ap.add_argument("--path", default="auto", choices=["auto", "ray", "column"])
    ap.add_argument("--ref-budget", type=float, default=15.0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--partition", default="replicas", choices=["replicas", "views"],
                    help="replicas: every rank runs the whole workload (weak scaling, the "
                         "default); views: the workload's views are sharded over the ranks "
                         "and the backward's volume is all-reduced (strong scaling)")
    ap.add_argument("--plan-options", type=json.loads, default=None,
                    help="work-layout options of the plan as JSON, e.g. "
                         "'{\"backward_staged\": \"direct\"}' (ctp_plan_options)")
    ap.add_argument("--no-per-workload", action="store_true",
                    help="skip the forward / backward timings of the other four workloads")
    ap.add_argument("--op", default="siddon", choices=["siddon", "fdk", "geometry"],
                    help="siddon: the projector pair (default); fdk: the analytical "
                         "filtered backprojection on the same workload; geometry: the "
                         "projection's geometry gradients")
    args = ap.parse_args(argv)
    if args.warmup < 3:
        ap.error("--warmup must be at least 3")
    w = ci.get(args.config)
    if args.views is not None:
        import dataclasses
        w = dataclasses.replace(w, n_views=args.views, name=f"{w.name}_views{args.views}")
    world, rank, local = dist_setup(args.gpus)
    try:
        if args.impl == "reference":
            return run_reference(args, w, world, rank)
        if args.op == "fdk":
            return run_fdk(args, w, world, rank, local)
        if args.op == "geometry":
            return run_geometry(args, w, world, rank, local)
        if args.partition == "views":
            return run_partitioned(args, w, world, rank, local)
        return run_gpu(args, w, world, rank, local)
    finally:
        if world > 1:
            import torch.distributed as dist
            dist.destroy_process_group()


if __name__ == "__main__":
    sys.exit(main())
