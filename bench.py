#!/usr/bin/env python3
"""float_vif throughput on GB300: frame pairs per second (4 scales).

A step is one pass of the whole path (taps, decimation to scales 1..3, the
statistic and terms at every scale, row sums, per-scale sums and scores) over
one batch of the workload's frames, through libfvif's C ABI.

  value  device-resident inputs (uploaded before the timed region),
         fvif_score_async on one stream, CUDA events around K steps.
  e2e    page-locked host inputs through fvif_score_host: the host->device
         copies of every step's frames and the device->host read of the
         scores are inside the timed region.
  roofline  the dominant kernel (the scale-0 statistic launch), timed by the
         library's own events around each launch on the launching stream.
  cpu_baseline  the CPU oracle (test infrastructure, never tuned) on a
         bounded sample of the same workload, frame-parallel on host cores.

``--impl reference`` times the oracle alone as the reference arm.
Multi-GPU (torchrun): every rank scores its own batch (weak scaling, no
data-path collective); the step time is the maximum over ranks.
"""
from __future__ import annotations

import argparse
import gc
import hashlib
import json
import os
import re
import subprocess
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

from vmaf_float_vif_gb300 import synthetic as S  # noqa: E402

PEAKS_PATH = os.path.join(ROOT, "MEASURED_PEAKS.json")
TRAFFIC_PATH = os.path.join(ROOT, "profiles", "stats_scale0_traffic.json")
KERNEL_SOURCES = ["fvif_kernels.cuh", "fvif_dispatch.cuh", "fvif_stats_u8.cu",
                  "fvif_stats_u16.cu", "fvif_internal.h"]
SMS = 152
FP32_LANES_PER_SM = 128
FALLBACK_HBM_GBS = 6800.0

WORKLOADS = {
    # name: (case, frames per step, kernelscale)
    "c5_4k_10b": ("c5_4k_10b", 240, 1.0),
    "c5_4k_10b_ks0.5": ("c5_4k_10b", 240, 0.5),
    "c5_4k_10b_ks2": ("c5_4k_10b", 240, 2.0),
    "c4_4k_8b": ("c4_4k_8b", 20, 1.0),
    "c2_1080p_10b": ("c2_checker_1px_10b", 240, 1.0),
    "c3_1080p_16b": ("c3_bright_1080p_16b", 240, 1.0),
    "c1_576x324_8b": ("c1_576x324_8b", 960, 1.0),
}


def describe(name, frames_override=None):
    case_name, frames, ks = WORKLOADS[name]
    frames = frames_override or frames
    c = S.CASES[case_name]
    return ("%s: %dx%d %d-bit luma pairs, %d frames per step, "
            "kernelscale %g, sigma_nsq %g" % (case_name, c.w, c.h, c.bitdepth,
                                              frames, ks, c.nsq))


def make_inputs(name, frames_override=None):
    case_name, frames, _ = WORKLOADS[name]
    frames = frames_override or frames
    case = S.CASES[case_name]
    if case.frames >= frames:
        return case, case.batch(range(frames))
    return case, S.streamed_batch(case, frames)


def dist_env():
    return (int(os.environ.get("RANK", "0")),
            int(os.environ.get("LOCAL_RANK", "0")),
            int(os.environ.get("WORLD_SIZE", "1")))


def max_over_ranks(x: float, world: int) -> float:
    """The largest value of x over all ranks (the job's step time is its
    slowest rank's).  The only collective of a multi-GPU run besides the
    barriers; frame pairs never leave their GPU."""
    if world <= 1:
        return x
    import torch
    import torch.distributed as dist
    dev = "cuda" if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([x], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_throughput(frames_per_rank: int, steps: int, world: int,
                   seconds: float) -> float:
    """Whole-job frame pairs per second: every rank scores its own
    frames_per_rank each step (weak scaling)."""
    return frames_per_rank * steps * world / seconds


# ---------------------------------------------------------------------------
# clocks during the timed region


class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,"
              "clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,"
              "clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,"
              "clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.lines = []

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu),
                 "--query-gpu=" + self.FIELDS, "--format=csv,noheader,nounits",
                 "-lms", "200"], stdout=subprocess.PIPE,
                stderr=subprocess.DEVNULL, text=True)
            self.thread = threading.Thread(target=self._read, daemon=True)
            self.thread.start()
        except OSError:
            self.proc = None
        return self

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def __exit__(self, *exc):
        if self.proc:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
            self.thread.join(timeout=2)

    def summary(self):
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown",
                 "sw_power_cap"]
        for line in self.lines:
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                mx.append(float(parts[2]))
            except ValueError:
                continue
            for n, v in zip(names, parts[5:9]):
                if v.lower() == "active":
                    reasons.add(n)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [],
                    "samples": 0}
        return {"sm_mhz": float(np.median(sm)), "sm_max_mhz": max(mx),
                "reasons": sorted(reasons), "samples": len(sm)}


# ---------------------------------------------------------------------------
# CPU oracle timing


def oracle_rate(case, ref, dist, ks, frames_wanted, threads):
    import oracle
    oracle.build()
    oracle.lib()
    n = min(frames_wanted, ref.shape[0])
    t0 = time.perf_counter()
    oracle.score(ref[:n], dist[:n], case.bitdepth, ks, case.nsq,
                 threads=threads)
    dt = time.perf_counter() - t0
    return n / dt, n, dt


def host_cores():
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:
        return os.cpu_count() or 1


# ---------------------------------------------------------------------------


def source_hash(names):
    """Hash of the named CUDA sources with comments and whitespace removed:
    it changes with the code the counters were taken on, not with its
    comments."""
    h = hashlib.sha256()
    for n in names:
        with open(os.path.join(ROOT, "vmaf_float_vif_gb300", "csrc", n)) as f:
            text = f.read()
        text = re.sub(r"/\*.*?\*/", " ", text, flags=re.S)
        text = re.sub(r"//[^\n]*", " ", text)
        h.update(" ".join(text.split()).encode())
    return h.hexdigest()[:16]


def kernel_hash():
    return source_hash(KERNEL_SOURCES)


def load_traffic(workload, frames_per_launch):
    """DRAM bytes of one scale-0 statistic launch of frames_per_launch frames,
    from a committed ncu summary taken on the current kernel sources.  The
    capture holds fewer frames than a full launch; the traffic of a launch
    grows in proportion to its frames (each frame is read once), so it is
    scaled by the frame count."""
    try:
        with open(TRAFFIC_PATH) as f:
            t = json.load(f)
    except (OSError, ValueError):
        return None
    if t.get("kernel_hash") != kernel_hash():
        return None
    cap = t.get("captures", {}).get(workload)
    if not cap or not cap.get("frames"):
        return None
    return ((cap["dram_bytes_read"] + cap["dram_bytes_write"]) *
            frames_per_launch / cap["frames"])


def chunked_copy_control(pr, pd, frame_elems: int, chunk: int = 16,
                         reps: int = 3):
    """The host path's copy pattern with no kernels: the same page-locked
    input buffers copied to the device in chunks of ``chunk`` frames (ref
    then dist, one copy each per chunk) on one stream, as a whole step.
    Returns (median ms per step, GB/s)."""
    import torch
    fr, fd = pr.view(-1), pd.view(-1)
    n = fr.numel() // frame_elems
    dev = torch.empty(2 * chunk * frame_elems, dtype=fr.dtype, device="cuda")
    st = torch.cuda.Stream()
    times = []
    for _ in range(reps + 1):
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        with torch.cuda.stream(st):
            e0.record(st)
            for f0 in range(0, n, chunk):
                k = min(chunk, n - f0) * frame_elems
                a = f0 * frame_elems
                dev[:k].copy_(fr[a:a + k], non_blocking=True)
                dev[chunk * frame_elems:chunk * frame_elems + k].copy_(
                    fd[a:a + k], non_blocking=True)
            e1.record(st)
        st.synchronize()
        times.append(e0.elapsed_time(e1))
    times = sorted(times[1:])
    ms = times[len(times) // 2]
    nbytes = (pr.numel() + pd.numel()) * pr.element_size()
    return ms, nbytes / (ms / 1e3) / 1e9


def host_breakdown(t, wall_ms: float, nbytes: int):
    """Where one fvif_score_host call spent its time, from the library's
    per-chunk events (fvif_profile_host): the copies' busy time and rate,
    the copy stream's idle gaps between chunks, how long chunks waited on
    a busy lane after arriving, the device span, the host's enqueue time
    what the call spent outside the device span, and whether the library
    saw every chunk's inputs as page-locked."""
    c0, c1, s0, s1, h0, h1, locked = (t[:, k] for k in range(7))
    copy_ms = float(np.sum(c1 - c0))
    return {"copy_ms": round(copy_ms, 2),
            "copy_gbs": round(nbytes / (copy_ms / 1e3) / 1e9, 1),
            "copy_idle_ms": round(float(np.sum(np.maximum(
                0.0, c0[1:] - c1[:-1]))), 2),
            "lane_busy_after_copy_ms": round(float(np.sum(s0 - c1)), 2),
            "device_ms": round(float(np.max(s1)), 2),
            "enqueue_ms": round(float(h1[-1]), 2),
            "outside_device_ms": round(wall_ms - float(np.max(s1)), 2),
            "inputs_page_locked": bool(np.all(locked == 1.0))}


def host_link_gbs(copies: int = 8):
    """Host-to-device bandwidth of this process's GPU for page-locked
    memory: 1 GiB copies timed with CUDA events, as (min, median, max) GB/s.
    The spread matters: on a shared host the link's bandwidth drops for
    stretches of time."""
    import torch
    n = 1 << 30
    h = torch.empty(n, dtype=torch.uint8).pin_memory()
    d = torch.empty(n, dtype=torch.uint8, device="cuda")
    d.copy_(h, non_blocking=True)
    torch.cuda.synchronize()
    rates = []
    for _ in range(copies):
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e0.record()
        d.copy_(h, non_blocking=True)
        e1.record()
        torch.cuda.synchronize()
        rates.append(n / (e0.elapsed_time(e1) / 1e3) / 1e9)
    del h, d
    rates.sort()
    return rates[0], rates[len(rates) // 2], rates[-1]


def stats_ops_per_pixel(ntaps: int) -> int:
    """Algorithmic fp32 operations of the statistic per pixel: a multiply and
    an add per tap for five quantities in two passes (20 N), and about 60 for
    the products x*x, y*y, x*y, the statistic with its guards, the two terms
    and the two log2 evaluations."""
    return 20 * ntaps + 60


def frame_ops(w: int, h: int, taps) -> int:
    """Algorithmic fp32 operations of one frame pair over the four scales:
    the statistic at every pixel of every scale (stats_ops_per_pixel), and
    3 N_s operations per pixel of plane s-1 for each decimation into scale s
    (about 4.2e9 for a 4K frame pair at kernelscale 1)."""
    ops = 0
    ws, hs = w, h
    for s in range(4):
        if s > 0:
            ops += 3 * taps[s] * ws * hs
            ws, hs = ws // 2, hs // 2
        ops += ws * hs * stats_ops_per_pixel(taps[s])
    return ops


def measured_alu_peak(local_rank: int, iters: int = 800_000, reps: int = 3):
    """The measured rate of separately rounded fp32 multiplies and adds on
    this GPU (fvif_alu_probe: independent mul-then-add chains in every lane,
    scalar and packed two-lane forms, about 50 ms per launch, best of
    reps), with the SM clock sampled while it runs.  The larger of the two
    forms is the roofline's peak."""
    import vmaf_float_vif_gb300 as fv
    fv.fvif_alu_probe(False, iters // 8)
    fv.fvif_alu_probe(True, iters // 8)
    best = {}
    with ClockSampler(local_rank) as clk:
        for packed in (False, True):
            rates = []
            for _ in range(reps):
                ops, ms = fv.fvif_alu_probe(packed, iters)
                rates.append(ops / (ms / 1e3) / 1e12)
            best["packed" if packed else "scalar"] = max(rates)
    c = clk.summary()
    return {"tops": max(best.values()), "scalar_tops": best["scalar"],
            "packed_tops": best["packed"], "clocks": c}


def also_line(name, args, alu, inputs=None):
    """Device-resident throughput of another workload (same timing as the
    main line), with its own ALU roofline for the scale-0 statistic launch
    and the whole step, its clocks, and the oracle on a sample of it."""
    import torch
    import vmaf_float_vif_gb300 as fv
    case, (ref, dist_np) = inputs if inputs else make_inputs(name)
    _, frames, ks = WORKLOADS[name]

    def as_dev(a):
        return torch.from_numpy(a.view(np.int16) if a.dtype == np.uint16
                                else a).to("cuda")
    r, d = as_dev(ref), as_dev(dist_np)
    out = torch.empty(4 * frames, dtype=torch.float64, device="cuda")
    stream = torch.cuda.Stream()
    with fv.Context(case.w, case.h, case.bitdepth, ks, case.nsq) as ctx:
        ctx.set_stream(stream)
        taps = [len(ctx.taps(s)) for s in range(4)]
        chunk = ctx.chunk_frames
        for _ in range(args.warmup):
            ctx.score_async(r, d, out)
        torch.cuda.synchronize()
        ctx.profile(True)
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        with ClockSampler(int(os.environ.get("LOCAL_RANK", "0"))) as clocks:
            e0.record(stream)
            for _ in range(args.steps):
                ctx.score_async(r, d, out)
            e1.record(stream)
            torch.cuda.synchronize()
        prof = ctx.profile_read()
        ctx.profile(False)
    ms = e0.elapsed_time(e1) / args.steps
    del r, d, out
    st0_ms, st0_n = prof["stats_scale0"]
    launches_step = -(-frames // chunk)
    frames_launch = frames / launches_step
    ops_launch = frames_launch * case.w * case.h * stats_ops_per_pixel(taps[0])
    achieved = ops_launch / (st0_ms / max(1, st0_n) / 1e3) / 1e12
    step_ops = frames * frame_ops(case.w, case.h, taps)
    traffic = load_traffic(name, frames_launch)
    line = {"workload": describe(name), "value": frames / (ms / 1e3),
            "unit": "frame-pairs/s", "ms_per_step": ms,
            "frames_per_step": frames, "chunk_frames": chunk, "taps": taps,
            "roofline": {
                "kernel": "stats_kernel, scale 0 (%d taps), %.4g frames per "
                          "launch" % (taps[0], frames_launch),
                "bound": "alu", "achieved": achieved, "peak": alu["tops"],
                "unit": "TFLOP/s", "frac": achieved / alu["tops"],
                "peak_note": "of measured (fvif_alu_probe)",
                "launch_ms": st0_ms / max(1, st0_n),
                "traffic": traffic,
                "traffic_note": traffic_note(traffic, TRAFFIC_PATH, True),
                "step_achieved": step_ops / (ms / 1e3) / 1e12,
                "step_frac": step_ops / (ms / 1e3) / 1e12 / alu["tops"]},
            "clocks": clocks.summary()}
    if not args.no_cpu_baseline:
        cores = host_cores()
        rate, n, dt = oracle_rate(case, ref, dist_np, ks, cores, cores)
        line["cpu_baseline"] = {
            "value": rate, "unit": "frame-pairs/s", "cores": cores,
            "kind": "oracle",
            "sample": "%d frames of the workload, one per host thread, "
                      "%.1f s wall" % (n, dt)}
    return line


def run_ours(args):
    import torch
    import vmaf_float_vif_gb300 as fv

    rank, local_rank, world = dist_env()
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl")
    torch.cuda.set_device(local_rank)
    fv.build()

    case, (ref, dist_np) = make_inputs(args.workload, args.frames)
    _, frames, ks = WORKLOADS[args.workload]
    frames = args.frames or frames
    bpp = case.bytes_per_pair

    def as_dev(a):
        if a.dtype == np.uint16:
            a = a.view(np.int16)
        return torch.from_numpy(a).to("cuda")

    r_dev, d_dev = as_dev(ref), as_dev(dist_np)
    out = torch.empty(4 * frames, dtype=torch.float64, device="cuda")
    stream = torch.cuda.Stream()
    ctx = fv.Context(case.w, case.h, case.bitdepth, ks, case.nsq)
    ctx.set_stream(stream)
    n0 = len(ctx.taps(0))
    chunk = ctx.chunk_frames

    def barrier():
        if world > 1:
            import torch.distributed as dist
            dist.barrier()

    with torch.cuda.stream(stream):
        for _ in range(args.warmup):
            ctx.score_async(r_dev, d_dev, out)
    torch.cuda.synchronize()
    alu = measured_alu_peak(local_rank)

    ctx.profile(True)
    start = torch.cuda.Event(enable_timing=True)
    stop = torch.cuda.Event(enable_timing=True)
    barrier()
    torch.cuda.synchronize()
    # no interpreter garbage-collection pass inside a timed region: a full
    # pass over the objects torch and the input generation created stalls
    # the launching thread for a few hundred ms
    gc.collect()
    gc.disable()
    with ClockSampler(local_rank) as clocks:
        start.record(stream)
        for _ in range(args.steps):
            ctx.score_async(r_dev, d_dev, out)
        stop.record(stream)
        torch.cuda.synchronize()
    gc.enable()
    barrier()
    ms_total = start.elapsed_time(stop)
    prof = ctx.profile_read()
    ctx.profile(False)
    # one chunk alone (after the timed region): its launches share the GPU
    # with nothing, which gives the dominant kernel's standalone duration
    n_solo = min(ctx.chunk_frames, frames)
    out_solo = torch.empty(4 * n_solo, dtype=torch.float64, device="cuda")
    ctx.profile(True)
    for _ in range(3):
        ctx.score_async(r_dev[:n_solo], d_dev[:n_solo], out_solo)
    solo = ctx.profile_read()
    ctx.profile(False)
    solo_ms = solo["stats_scale0"][0] / max(1, solo["stats_scale0"][1])
    scores = out.cpu().numpy().reshape(-1, 4)
    if not np.all(np.isfinite(scores)):
        raise RuntimeError("non-finite scores")

    ms_total = max_over_ranks(ms_total, world)
    ms_step = ms_total / args.steps
    value = job_throughput(frames, args.steps, world, ms_total / 1e3)

    # e2e: host buffers, copies inside the timed region
    e2e = None
    if not args.no_e2e:
        # the inputs in page-locked buffers from the library's own host
        # allocator (fvif_host_alloc: huge-page aligned and registered)
        bufs = [fv.HostBuffer(ref.nbytes), fv.HostBuffer(dist_np.nbytes)]
        hr = bufs[0].array(ref.shape, ref.dtype)
        hd = bufs[1].array(dist_np.shape, dist_np.dtype)
        np.copyto(hr, ref)
        np.copyto(hd, dist_np)

        def as_torch(a):
            return torch.from_numpy(a.view(np.int16) if a.dtype == np.uint16
                                    else a)
        pr, pd = as_torch(hr), as_torch(hd)
        h2d_bytes = int(ref.nbytes + dist_np.nbytes)
        link = host_link_gbs()
        control = chunked_copy_control(pr, pd, case.w * case.h)
        ctx.set_stream(None)

        def e2e_run(r_host, d_host, steps):
            """steps timed fvif_score_host calls (after warm-up), with the
            library's per-chunk events on; each step's table is read
            between steps, outside the step's own time."""
            for _ in range(max(1, args.warmup)):
                ctx.score_host(r_host, d_host)
            barrier()
            torch.cuda.synchronize()
            ctx.profile(True)
            gc.collect()
            gc.disable()
            times, tables = [], []
            for _ in range(steps):
                ts = time.perf_counter()
                res = ctx.score_host(r_host, d_host)  # after the d2h read
                times.append(1e3 * (time.perf_counter() - ts))
                tables.append(host_breakdown(ctx.profile_host(), times[-1],
                                             h2d_bytes))
            gc.enable()
            ctx.profile(False)
            barrier()
            return res, times, tables

        host_scores, step_ms, parts = e2e_run(hr, hd, args.e2e_steps)
        wall = max_over_ranks(sum(step_ms) / 1e3, world)
        control_after = chunked_copy_control(pr, pd, case.w * case.h)
        link_after = host_link_gbs()
        if not np.array_equal(host_scores, scores):
            raise RuntimeError("fvif_score_host and fvif_score_async differ")
        # the same calls from buffers pinned by torch (cudaHostAlloc), for
        # comparison: their copy rate is what the host allocator avoids
        # (one process only: N ranks on one host would pin N more copies)
        torch_pinned = None
        if world == 1:
            tr = torch.from_numpy(ref.view(np.int16)
                                  if ref.dtype == np.uint16 else ref
                                  ).pin_memory()
            td = torch.from_numpy(dist_np.view(np.int16)
                                  if dist_np.dtype == np.uint16
                                  else dist_np).pin_memory()
            alt_scores, alt_ms, alt_parts = e2e_run(
                tr.numpy().view(ref.dtype), td.numpy().view(dist_np.dtype),
                args.e2e_steps)
            if not np.array_equal(alt_scores, scores):
                raise RuntimeError("fvif_score_host differs on torch buffers")
            del tr, td
            torch_pinned = {
                "value": job_throughput(frames, args.e2e_steps, 1,
                                        sum(alt_ms) / 1e3),
                "step_ms": [round(t, 2) for t in alt_ms],
                "copy_gbs": [b["copy_gbs"] for b in alt_parts],
                "note": "the same fvif_score_host calls from buffers made "
                        "by torch's pin_memory (cudaHostAlloc)"}
        e2e = {"value": job_throughput(frames, args.e2e_steps, world, wall),
               "unit": "frame-pairs/s",
               "h2d_bytes_per_step": h2d_bytes,
               "d2h_bytes_per_step": int(scores.nbytes),
               "ms_per_step": 1e3 * wall / args.e2e_steps,
               "api": "fvif_score_host (inputs in fvif_host_alloc buffers)",
               "step_ms": [round(t, 2) for t in step_ms],
               "median_step_ms": float(np.median(step_ms)),
               "value_at_median_step": job_throughput(
                   frames, 1, world, float(np.median(step_ms)) / 1e3),
               "breakdown": parts,
               "breakdown_note": "per timed step, from the library's "
                                 "per-chunk events (fvif_profile_host): "
                                 "copy busy time and rate, idle gaps of the "
                                 "copy stream between chunks, time chunks "
                                 "waited on a busy lane after arriving, "
                                 "device span, host enqueue time, and wall "
                                 "time outside the device span",
               "copy_control": {
                   "before_ms": round(control[0], 2),
                   "before_gbs": round(control[1], 1),
                   "after_ms": round(control_after[0], 2),
                   "after_gbs": round(control_after[1], 1),
                   "note": "the same host buffers copied in chunks of 16 "
                           "frames with no kernels, one stream, median of 3 "
                           "whole steps"},
               "torch_pinned": torch_pinned,
               "h2d_link_gbs": {
                   "before": [round(x, 1) for x in link],
                   "after": [round(x, 1) for x in link_after]},
               "link_floor_ms": 1e3 * (ref.nbytes + dist_np.nbytes) / 1e9 /
                                link[2],
               "link_note": "plain page-locked 1 GiB host-to-device copies "
                            "(min, median, max of 8) just before and just "
                            "after the e2e region; a step cannot finish faster "
                            "than its input bytes over the link at its "
                            "best"}
        del pr, pd, hr, hd
        for b in bufs:
            b.close()

    if rank != 0:
        ctx.close()
        if world > 1:
            import torch.distributed as dist
            dist.destroy_process_group()
        return

    peaks = {}
    try:
        with open(PEAKS_PATH) as f:
            peaks = json.load(f)
    except (OSError, ValueError):
        pass
    hbm_peak = peaks.get("hbm_gbs")
    hbm_src = "of measured" if hbm_peak else "of fallback"
    hbm_peak = hbm_peak or FALLBACK_HBM_GBS
    clk = clocks.summary()
    sm_max = clk.get("sm_max_mhz") or peaks.get("sm_max_mhz") or 2070.0

    taps = [len(ctx.taps(s)) for s in range(4)]
    step_ops = frames * frame_ops(case.w, case.h, taps)
    st0_ms, st0_n = prof["stats_scale0"]
    launches_total = sum(n for _, n in prof.values())
    px0 = case.w * case.h
    # frames per scale-0 launch: full chunks, the last one partial
    launches_step = -(-frames // chunk)
    frames_launch = frames / launches_step
    ops_launch = frames_launch * px0 * stats_ops_per_pixel(n0)
    ops_solo = n_solo * px0 * stats_ops_per_pixel(n0)
    avg_ms = st0_ms / max(1, st0_n)
    achieved = ops_launch / (avg_ms / 1e3) / 1e12
    alu_derived = SMS * FP32_LANES_PER_SM * sm_max * 1e6 / 1e12
    alu_peak = alu["tops"]
    traffic = load_traffic(args.workload, frames_launch)
    kernel_shares = {k: {"ms": v[0], "launches": v[1],
                         "share": v[0] / max(1e-9, sum(x[0] for x in
                                                       prof.values()))}
                     for k, v in prof.items()}

    line = {
        "metric": "float_vif frame-pairs/s, 4 scales (%dx%d %d-bit)" %
                  (case.w, case.h, case.bitdepth),
        "value": value,
        "unit": "frame-pairs/s",
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": ms_step,
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "f32",
        "data": "synthetic",
        "config": {
            "workload": describe(args.workload, args.frames),
            "frames_per_step": frames,
            "chunk_frames": chunk,
            "taps": taps,
            "l2": "no flush: inputs %.2f GB per step exceed the 129 MB L2" %
                  (frames * bpp / 1e9),
            "hbm_fraction_algorithmic": value / world * bpp / 1e9 / hbm_peak,
            "hbm_fraction_note": "input bytes only (%d B per pair) against "
                                 "%.1f GB/s %s" % (bpp, hbm_peak, hbm_src),
            "kernels": kernel_shares,
            "kernels_note": "summed event durations of each kind's launches "
                            "on their own streams over the timed steps; the "
                            "scale-0 stream and the two lanes overlap, and a "
                            "low-priority launch's duration includes the time "
                            "it waits for SMs, so these overlap and exceed "
                            "the step (serialised shares: the ncu launch "
                            "list under profiles/)",
        },
        "roofline": {
            "kernel": "stats_kernel, scale 0 (%d taps), %.4g frames per "
                      "launch (chunks of %d)" % (n0, frames_launch, chunk),
            "bound": "alu",
            "achieved": achieved,
            "peak": alu_peak,
            "unit": "TFLOP/s",
            "frac": achieved / alu_peak,
            "traffic": traffic,
            "traffic_note": traffic_note(traffic, TRAFFIC_PATH, True),
            "per_unit": "%d fp32 ops per pixel (20 N + 60: a multiply and "
                        "an add per tap for five quantities in two passes, "
                        "plus the products, statistic, terms and log2)"
                        % stats_ops_per_pixel(n0),
            "launch_ms": avg_ms,
            "peak_note": "of measured: fvif_alu_probe, separately rounded "
                         "fp32 multiply-then-add chains in every lane (best "
                         "of scalar %.2f and packed two-lane %.2f T ops/s, "
                         "SM clock median %s MHz while it ran); derived "
                         "%d SMs x %d lanes x %.0f MHz = %.2f T" % (
                             alu["scalar_tops"], alu["packed_tops"],
                             alu["clocks"].get("sm_mhz"), SMS,
                             FP32_LANES_PER_SM, sm_max, alu_derived),
            "frac_of_derived": achieved / alu_derived,
            "launch_note": "events on the launching stream; consecutive chunks "
                           "run on two streams, so a launch shares the GPU "
                           "with the other chunk's smaller kernels",
            "solo_launch_ms": solo_ms,
            "solo_achieved": ops_solo / (solo_ms / 1e3) / 1e12,
            "solo_frac": ops_solo / (solo_ms / 1e3) / 1e12 / alu_peak,
            "solo_note": "the same launch with no other chunk in flight "
                         "(one chunk scored alone after the timed "
                         "region, events on its stream)",
            "step_achieved": step_ops / (ms_step / 1e3) / 1e12,
            "step_frac": step_ops / (ms_step / 1e3) / 1e12 / alu_peak,
            "step_note": "all algorithmic fp32 operations of a step (%.3g "
                         "per frame pair: the statistic at 20 N + 60 per pixel "
                         "of each scale, each decimation at 3 N per pixel of "
                         "its source plane) / step time" % (step_ops / frames),
        },
        "gpu_launches": int(launches_total),
        "clocks": clk,
    }
    ctx.close()
    also = [a for a in (args.also or "").split(",") if a and
            a != args.workload]
    if also:
        line["also"] = {}
        for name in also:
            same = (WORKLOADS[name][0] == WORKLOADS[args.workload][0] and
                    WORKLOADS[name][1] == frames)
            line["also"][name] = also_line(
                name, args, alu,
                inputs=(case, (ref, dist_np)) if same else None)
    if not args.no_ssim:
        line["ssim_decimate"] = ssim_decimate_lines(
            args, hbm_peak, hbm_src, cpu_baseline=not args.no_cpu_baseline)
    if e2e:
        line["e2e"] = e2e
    if not args.no_cpu_baseline:
        cores = host_cores()
        rate, n, dt = oracle_rate(case, ref, dist_np, ks, cores, cores)
        line["cpu_baseline"] = {
            "value": rate, "unit": "frame-pairs/s", "cores": cores,
            "kind": "oracle",
            "sample": "%d frames of the workload, one per host thread, "
                      "%.1f s wall" % (n, dt)}
    print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


# float_ssim auto-scale decimation: name -> (w, h, bitdepth, frames per launch)
SSIM_WORKLOADS = {
    "ssim_dec_4k_8b": (3840, 2160, 8, 64),
    "ssim_dec_720p_8b": (1280, 720, 8, 512),
}
SSIM_TRAFFIC_PATH = os.path.join(ROOT, "profiles", "ssim_decimate_traffic.json")
SSIM_KERNEL_SOURCES = ["fssim_kernels.cuh", "fssim_u8.cu", "fssim_u16.cu",
                       "fssim_api.cu"]


def ssim_kernel_hash():
    return source_hash(SSIM_KERNEL_SOURCES)


def traffic_note(value, path, scaled):
    rel = os.path.relpath(path, ROOT)
    if value is None:
        return ("null: %s holds no ncu capture taken on the current kernel "
                "sources" % rel)
    return ("dram__bytes_read.sum + dram__bytes_write.sum of one ncu capture "
            "(%s)%s" % (rel, ", scaled to this launch's frames" if scaled
                        else ""))


def ssim_traffic(name):
    try:
        with open(SSIM_TRAFFIC_PATH) as f:
            t = json.load(f)
    except (OSError, ValueError):
        return None
    if t.get("kernel_hash") != ssim_kernel_hash():
        return None
    return t.get("per_launch_bytes", {}).get(name)


def ssim_decimate_lines(args, hbm_peak, hbm_src, cpu_baseline=True):
    """float_ssim's auto-scale decimation of frame pairs (a second workload
    of the library): one fssim_decimate launch of F frame pairs per step,
    device-resident inputs larger than L2, CUDA events on the launching
    stream; the HBM roofline counts the input samples read once and the
    fp32 planes written once."""
    import torch
    import vmaf_float_vif_gb300 as fv
    out = {}
    for name, (w, h, bd, frames) in SSIM_WORKLOADS.items():
        case = S.video_case(w, h, bd, frames=8, seed=21)
        ref, dist_np = S.streamed_batch(case, frames, distinct=8)

        def as_dev(a):
            return torch.from_numpy(a.view(np.int16) if a.dtype == np.uint16
                                    else a).to("cuda")
        r, d = as_dev(ref), as_dev(dist_np)
        scale = fv.fssim_auto_scale(w, h)
        sw, sh = fv.fssim_decimated_size(w, h, scale)
        ro = torch.empty((frames, sh, sw), dtype=torch.float32, device="cuda")
        do = torch.empty_like(ro)
        stream = torch.cuda.Stream()
        with torch.cuda.stream(stream):
            for _ in range(max(3, args.warmup)):
                fv.fssim_decimate(r, d, w, h, bd, 0, ro, do, stream)
        torch.cuda.synchronize()
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for _ in range(args.steps):
            fv.fssim_decimate(r, d, w, h, bd, 0, ro, do, stream)
        e1.record(stream)
        torch.cuda.synchronize()
        ms = e0.elapsed_time(e1) / args.steps
        B = 1 if bd == 8 else 2
        per_pair = 2 * w * h * B + 2 * sw * sh * 4
        achieved = frames * per_pair / (ms / 1e3) / 1e9
        entry = {
            "workload": "%dx%d %d-bit, auto scale %d -> %dx%d, %d frame "
                        "pairs per launch (%.2f GB, larger than L2)" %
                        (w, h, bd, scale, sw, sh, frames,
                         frames * 2 * w * h * B / 1e9),
            "value": frames / (ms / 1e3), "unit": "frame-pairs/s",
            "ms_per_launch": ms,
            "roofline": {
                "bound": "hbm", "achieved": achieved, "peak": hbm_peak,
                "unit": "GB/s", "frac": achieved / hbm_peak,
                "peak_note": hbm_src,
                "traffic": ssim_traffic(name),
                "traffic_note": traffic_note(ssim_traffic(name),
                                             SSIM_TRAFFIC_PATH, False),
                "per_unit": "%d bytes per frame pair (samples read once, "
                            "fp32 planes written once)" % per_pair,
            },
        }
        if cpu_baseline:
            import oracle
            cores = host_cores()
            n = min(frames, 2 * cores)
            t0 = time.perf_counter()
            oracle.ssim_decimate(ref[:n], dist_np[:n], bd, 0, threads=cores)
            dt = time.perf_counter() - t0
            entry["cpu_baseline"] = {
                "value": n / dt, "unit": "frame-pairs/s", "cores": cores,
                "kind": "oracle",
                "sample": "%d frame pairs of the workload over %d host "
                          "threads, %.1f s wall" % (n, cores, dt)}
        out[name] = entry
        del r, d, ro, do
        torch.cuda.empty_cache()
    return out


def run_ssim_only(args):
    import torch
    import vmaf_float_vif_gb300 as fv
    fv.build()
    torch.cuda.init()
    peaks = {}
    try:
        with open(PEAKS_PATH) as f:
            peaks = json.load(f)
    except (OSError, ValueError):
        pass
    hbm_peak = peaks.get("hbm_gbs")
    hbm_src = "of measured" if hbm_peak else "of fallback"
    lines = ssim_decimate_lines(args, hbm_peak or FALLBACK_HBM_GBS, hbm_src,
                                cpu_baseline=not args.no_cpu_baseline)
    print(json.dumps({"ssim_decimate": lines, "steps": args.steps,
                      "warmup": max(3, args.warmup)}), flush=True)


def run_reference(args):
    rank, _, world = dist_env()
    if rank != 0:
        return
    case, (ref, dist_np) = make_inputs_sample(args.workload)
    _, frames, ks = WORKLOADS[args.workload]
    cores = host_cores()
    per_step = min(cores, ref.shape[0])
    for _ in range(args.warmup):
        oracle_rate(case, ref, dist_np, ks, per_step, cores)
    t0 = time.perf_counter()
    for _ in range(args.steps):
        oracle_rate(case, ref, dist_np, ks, per_step, cores)
    wall = time.perf_counter() - t0
    value = per_step * args.steps / wall
    line = {
        "impl": "reference",
        "metric": "float_vif frame-pairs/s, 4 scales (%dx%d %d-bit)" %
                  (case.w, case.h, case.bitdepth),
        "value": value,
        "unit": "frame-pairs/s",
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": 1e3 * wall / args.steps,
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "f32",
        "data": "synthetic",
        "config": {"workload": describe(args.workload),
                   "frames_per_step": per_step,
                   "note": "each step scores a bounded sample of the "
                           "workload (one frame per host thread)"},
        "cpu_baseline": {"value": value, "unit": "frame-pairs/s",
                         "cores": cores, "kind": "oracle",
                         "sample": "%d frames per step" % per_step},
        "e2e": {"value": value, "unit": "frame-pairs/s",
                "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def make_inputs_sample(name):
    case_name, frames, _ = WORKLOADS[name]
    case = S.CASES[case_name]
    n = min(frames, max(1, host_cores()), 16)
    if case.frames >= n:
        return case, case.batch(range(n))
    return case, S.streamed_batch(case, n)


def main():
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=10)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", choices=sorted(WORKLOADS), default="c5_4k_10b")
    ap.add_argument("--frames", type=int, default=None,
                    help="frames per step (default: the workload's)")
    ap.add_argument("--e2e-steps", type=int, default=None,
                    help="timed fvif_score_host steps (default: --steps)")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-ssim", action="store_true",
                    help="skip the float_ssim decimation measurement")
    ap.add_argument("--ssim-only", action="store_true",
                    help="only the float_ssim decimation measurement (one "
                         "JSON line; the small case the decimation profiles "
                         "are captured on)")
    ap.add_argument("--also",
                    default=",".join(w for w in WORKLOADS
                                     if w != "c5_4k_10b"),
                    help="comma-separated other workloads timed "
                         "device-resident, each with its own roofline and "
                         "oracle baseline (\"\" = none; default: every "
                         "other workload)")
    args = ap.parse_args()
    if args.e2e_steps is None:
        args.e2e_steps = max(1, args.steps)
    for name in (args.also or "").split(","):
        if name and name not in WORKLOADS:
            ap.error("--also: unknown workload %r (choose from %s)" %
                     (name, ", ".join(sorted(WORKLOADS))))
    if args.warmup < 3 and args.impl == "ours":
        print("note: fewer than 3 warm-up steps", file=sys.stderr)
    if args.impl == "reference":
        run_reference(args)
    elif args.ssim_only:
        run_ssim_only(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
