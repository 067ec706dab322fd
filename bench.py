"""Benchmark of the training step of the tile-based 3D Gaussian splatting rasterizer.

One step = the whole hot path for one view: gs_preprocess, gs_bin_and_sort, gs_render_fwd,
gs_render_bwd_sqerr (the backward with the squared-error loss gradient image - target formed in the
kernel), gs_preprocess_bwd. The workload is the outdoor
scene: 1.6M Gaussians, 1297x840, SH degree 3, a 64-cluster mixture (seeded, synthetic).

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference] [--mode sm|direct|warp|adaptive]

The step is captured once into a CUDA graph (every kernel of the step, with the sort call that
does not synchronise) and each timed step is one replay; `--no-graph` times eager launches.

Prints one JSON line. `value` is the whole-job throughput in Mpix/s (pixels of all ranks' views
per second of the slowest rank), measured with CUDA events on the device with inputs resident;
`e2e` is the same metric through the C ABI's host-buffer entry point, gs_train_step_host: each
step copies its parameters and target in from pinned host memory and its parameter gradients,
loss and D back, inside the timed region; three step contexts on three streams take the steps in
turn, so a step's copies overlap its neighbours' compute and copies (the median of three timed
runs), and the serial
figure (one context) is reported beside it. `e2e.host_link` is the copy-engine bandwidth of the
host link measured alone (each direction, and both at once), the time one step's copies need at
that rate, and its fraction of the pipelined step. With N > 1 (torchrun) every rank runs an
independent replica of the step (the path needs no exchange within a view). `--impl reference`
times the float64 CPU oracle on the host cores instead, on a bounded sample of the same workload.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import re
import statistics
import subprocess
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "fwd+bwd ms/view and Mpix/s at 1.6M Gaussians 1297×840; bwd L2-atomic roofline %"
WORKLOADS = {
    0: "tiny: 2k Gaussians, 128x128, SH degree 0, one view per step",
    1: "object: 100k Gaussians, 800x800, SH degree 3, white background, one view per step",
    2: "outdoor: 1.6M Gaussians, 1297x840, SH degree 3, 64-cluster mixture, one view per step",
    3: "large: 3M Gaussians, 1959x1090, SH degree 3, 128-cluster mixture + shell, 8 views per step",
    4: "contention: 50k large Gaussians, 3840x2160, SH degree 0, one view per step",
}
CFG = 2  # the configuration the metric is quoted on (the default workload)
WORKLOAD = WORKLOADS[CFG]
PEAKS_PATH = os.path.join(ROOT, "MEASURED_PEAKS.json")
COUNTS_PATH = os.path.join(ROOT, "profiles", "workload_counts_outdoor.md")
TRAFFIC_PATH = os.path.join(ROOT, "profiles", "render_bwd_outdoor_1600k.md")
# the backward kernel's source and its device helpers: the ncu counters hold while these are unchanged
# (they are attached only to the default ADAPTIVE mode, whose 28-lane threshold they were taken with)
TRAFFIC_SOURCES = ("differentiable_gaussian_splatting_gs_gb300/csrc/render.cu",
                   "differentiable_gaussian_splatting_gs_gb300/csrc/gs_common.cuh")
# Algorithmic work of the backward raster. Every pixel's list is replayed back to front from its
# last contributor, and each replayed (pixel, Gaussian) pair needs its alpha: offsets 2, quadratic
# form 9, exponential 1, opacity product 1, clamp 1, threshold 1 = 15 FP32 operations. Each blended
# pair then needs its gradient: transmittance 4, colour gradient 3, alpha gradient 15, colour-behind
# update 6, opacity and geometry gradients 13 = 41.
BWD_FLOPS_ALPHA = 15
BWD_FLOPS_GRADIENT = 41


def parse_args():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--mode", default="adaptive", choices=["sm", "direct", "warp", "adaptive"])
    ap.add_argument("--threshold", type=int, default=0, help="adaptive threshold in lanes (0 = library default)")
    ap.add_argument("--staging", type=int, default=0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-extras", action="store_true", help="skip timing the update phase after the step")
    ap.add_argument("--no-graph", action="store_true",
                    help="time eager launches instead of one CUDA graph replay per step")
    ap.add_argument("--sync-sort", action="store_true",
                    help="time the step with the synchronising sort call (reads D on the host) instead of the "
                         "call that keeps the whole step enqueued ahead of the GPU")
    ap.add_argument("--config", type=int, default=CFG, choices=sorted(WORKLOADS),
                    help="workload; the default is the one the metric is quoted on")
    return ap.parse_args()


# ------------------------------------------------------------------------------------ helpers

class ClockSampler:
    """Samples SM clocks and throttle reasons with nvidia-smi while running."""

    QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.lines = []
        self.thread = None

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.QUERY}",
                                          "--format=csv,noheader,nounits", "-lms", "20"],
                                         stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.thread = threading.Thread(target=self._read, daemon=True)
            self.thread.start()
            self._wait_samples(1)  # a sample right before the timed region
        except OSError:
            self.proc = None
        return self

    def _wait_samples(self, k: int, timeout: float = 3.0):
        t0 = time.time()
        while len(self.lines) < k and time.time() - t0 < timeout and self.proc.poll() is None:
            time.sleep(0.005)

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def __exit__(self, *exc):
        if self.proc is not None:
            self._wait_samples(len(self.lines) + 1)  # and one right after it
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
            if self.thread:
                self.thread.join(timeout=2)

    def summary(self):
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            f = [x.strip() for x in ln.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                smax.append(float(f[2]))
            except ValueError:
                continue
            for name, val in zip(names, f[5:9]):
                if val.lower() == "active":
                    reasons.add(name)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(smax), "reasons": sorted(reasons),
                "samples": len(sm)}


def reduce_max(x: float, world: int, device=None) -> float:
    """Maximum of x over all ranks (the slowest rank's time); identity for one rank."""
    if world <= 1:
        return x
    import torch
    import torch.distributed as dist
    t = torch.tensor([x], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def throughput_mpix(world: int, pixels_per_step: int, ms_per_step: float) -> float:
    """Whole-job Mpix/s: every rank renders one step's views; the step takes the slowest rank's time."""
    return world * pixels_per_step / (ms_per_step / 1e3) / 1e6


def load_json(path):
    try:
        with open(path) as f:
            return json.load(f)
    except (OSError, ValueError):
        return None


def json_block(path):
    """The first ```json block of a markdown summary under profiles/."""
    try:
        text = open(path).read()
    except OSError:
        return None
    m = re.search(r"```json\s*(\{.*?\})\s*```", text, re.S)
    return json.loads(m.group(1)) if m else None


def source_hash(*rel_paths):
    h = hashlib.sha256()
    for p in rel_paths:
        with open(os.path.join(ROOT, p), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def flush_l2(flush):
    """Overwrites the L2 (a buffer larger than it), then keeps the GPU busy for about 0.1 ms so that
    the host enqueues what is timed next before the GPU reaches it: the events then bracket device
    time only, not the host's launch latency."""
    import torch
    flush.fill_(1.0)
    torch.cuda._sleep(200_000)


def host_link_gbs(host_buf, dev_buf, stream):
    """Copy-engine bandwidth between pinned host memory and the device, GB/s: host -> device and
    device -> host alone, and each direction while both run at once (two streams). host_buf is a
    pinned host tensor and dev_buf a device tensor of the same size; their contents are overwritten
    with each other's."""
    import torch
    dev = dev_buf.device
    back = torch.empty_like(host_buf).pin_memory()
    s1, s2 = torch.cuda.Stream(dev), torch.cuda.Stream(dev)
    nbytes = host_buf.numel() * host_buf.element_size()

    def best(fn, reps=4):
        fn()
        torch.cuda.synchronize()
        ts = []
        for _ in range(reps):
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            fn()
            e1.record(stream)
            torch.cuda.synchronize()
            ts.append(e0.elapsed_time(e1))
        return nbytes / min(ts) / 1e6

    def both():
        s1.wait_stream(stream)
        s2.wait_stream(stream)
        with torch.cuda.stream(s1):
            dev_buf.copy_(host_buf, non_blocking=True)
        with torch.cuda.stream(s2):
            back.copy_(dev_buf, non_blocking=True)
        stream.wait_stream(s1)
        stream.wait_stream(s2)

    with torch.cuda.stream(stream):
        return {"h2d_gbs": best(lambda: dev_buf.copy_(host_buf, non_blocking=True)),
                "d2h_gbs": best(lambda: back.copy_(dev_buf, non_blocking=True)),
                "both_gbs_each": best(both)}


def crop_camera(cam, frac_tiles_x: float, frac_tiles_y: float):
    """A tile-aligned window at the centre of the view (same tiles, same per-tile lists)."""
    import gs_scenes
    tx, ty = cam.tiles_x, cam.tiles_y
    wx, wy = max(1, int(round(tx * frac_tiles_x))), max(1, int(round(ty * frac_tiles_y)))
    x0, y0 = 16 * ((tx - wx) // 2), 16 * ((ty - wy) // 2)
    w, h = min(16 * wx, cam.width - x0), min(16 * wy, cam.height - y0)
    return gs_scenes.Camera(R=cam.R, t=cam.t, fx=cam.fx, fy=cam.fy, cx=cam.cx - x0, cy=cam.cy - y0, width=w,
                            height=h, bg=cam.bg), (x0, y0)


def oracle_sample(scene, frac_x: float, frac_y: float):
    """The oracle's whole step on a tile-aligned window of the view: preprocess of all Gaussians
    in the window's camera, then binning, render, backward and preprocess backward of the
    Gaussians that touch the window. Returns (pixels, seconds, description, threads)."""
    import gs_scenes
    import oracle
    cam, (x0, y0) = crop_camera(scene.cameras[0], frac_x, frac_y)
    t0 = time.perf_counter()
    pre = oracle.preprocess(scene.mean3d, scene.log_scale, scene.quat, scene.opacity_logit, scene.sh,
                            scene.sh_degree, cam)
    sel = pre["radius"] > 0
    sub = gs_scenes.Scene(name="window", mean3d=scene.mean3d[sel], log_scale=scene.log_scale[sel],
                          quat=scene.quat[sel], opacity_logit=scene.opacity_logit[sel], sh=scene.sh[sel],
                          sh_degree=scene.sh_degree, cameras=[cam],
                          targets=[scene.targets[0][:, y0:y0 + cam.height, x0:x0 + cam.width]])
    oracle.view_step(sub)
    dt = time.perf_counter() - t0
    desc = (f"float64 oracle, whole step on the central {cam.width}x{cam.height} tile-aligned window of the "
            f"view ({int(sel.sum())} Gaussians touch it; preprocess over all {scene.n})")
    return cam.width * cam.height, dt, desc, os.cpu_count()


def backward_roofline(counts: dict, peaks: dict, bwd_ms: float, dev, mode: str) -> dict:
    """Roofline line of the backward raster (the dominant kernel) at the outdoor scene.

    Algorithmic work, from the oracle's counts of the workload (profiles/workload_counts_outdoor.md):
    every (pixel, Gaussian) pair the method replays (each pixel's list back to front from its last
    contributor) needs its alpha evaluated, BWD_FLOPS_ALPHA FP32 operations; every blended pair
    needs its gradient, BWD_FLOPS_GRADIENT more. Peak: the device's SM count x 128 FP32 lanes x 2
    (fused multiply-add) x the measured maximum SM clock. The bound the pages name for this
    kernel, the L2 atomics, and its HBM traffic are reported beside it with their own fractions,
    and so is the resource that binds it (instruction issue, from the ncu capture)."""
    import torch
    sms = torch.cuda.get_device_properties(dev).multi_processor_count
    sm_mhz = float(peaks.get("sm_max_mhz", 2070.0))
    peak = sms * 128 * 2 * sm_mhz * 1e6 / 1e12
    flops = (counts["pairs_replayed_bwd"] * BWD_FLOPS_ALPHA + counts["pairs_blended"] * BWD_FLOPS_GRADIENT)
    ach = flops / (bwd_ms / 1e3) / 1e12
    hbm_peak = float(peaks.get("hbm_gbs", 6800.0))
    hbm_gbs = counts["bwd_bytes"] / (bwd_ms / 1e3) / 1e9
    traffic = l2_red = binding = None
    tr = json_block(TRAFFIC_PATH)
    # the counters hold while the kernel source and its launch defaults (the C ABI file) are unchanged
    if tr and tr.get("source_hash") == source_hash(*TRAFFIC_SOURCES) and mode == "adaptive":
        traffic = tr.get("dram_bytes_per_launch")
        if "l2_red_frac_of_peak" in tr:
            l2_red = {"sectors_per_launch": tr.get("l2_red_sectors_per_launch"),
                      "frac_of_peak": tr["l2_red_frac_of_peak"],
                      "source": "ncu, profiles/" + os.path.basename(TRAFFIC_PATH)}
        if "issue_active_frac" in tr:
            binding = {"resource": "instruction issue", "issue_active_frac": tr["issue_active_frac"],
                       "fma_pipe_frac": tr.get("fma_pipe_frac"),
                       "source": "ncu, profiles/" + os.path.basename(TRAFFIC_PATH)}
    return {"kernel": f"k_render_bwd ({mode} accumulation, bulk staging)", "bound": "alu", "achieved": ach,
            "peak": peak, "unit": "TFLOP/s", "frac": ach / peak, "traffic": traffic,
            "numerator": f"{BWD_FLOPS_ALPHA} FP32 operations per replayed (pixel, Gaussian) pair (its alpha) + "
                         f"{BWD_FLOPS_GRADIENT} per blended pair (its gradient), counts of the oracle",
            "algorithmic_flops": flops, "kernel_ms": bwd_ms,
            "peak_source": f"derived: {sms} SMs (device) x 128 FP32 lanes x 2 x {sm_mhz:.0f} MHz (measured max SM "
                           "clock, MEASURED_PEAKS.json)",
            "binding": binding,
            "l2_atomic": l2_red,
            "hbm": {"algorithmic_bytes": counts["bwd_bytes"], "achieved_gbs": hbm_gbs, "peak_gbs": hbm_peak,
                    "frac_of_measured": hbm_gbs / hbm_peak}}


def time_bwd_modes(api, bufs, cam, target, sh_degree, flush, stream, reps: int) -> dict:
    """The backward (gs_render_bwd_sqerr, as in the step) alone in each accumulation mode
    (gradient zeroing included), on the buffers of the step just run; L2 flushed before every
    launch; mean of `reps` launches per mode."""
    import torch
    image, t_final, n_contrib, _, ranges = bufs.image_buffers(cam.width, cam.height)
    out = {}
    for mode in ("direct", "warp", "adaptive", "sm"):
        opt = api.make_options(sh_degree, bwd_mode=mode)
        ts = []
        for it in range(reps + 2):
            flush_l2(flush)
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            api.gs_render_bwd_sqerr(bufs.proj, bufs.sort.vals, ranges, cam, opt, image, target, t_final, n_contrib,
                                    grad2d=bufs.grad2d)
            e1.record(stream)
            torch.cuda.synchronize()
            if it >= 2:
                ts.append(e0.elapsed_time(e1))
        out[f"{mode}_ms"] = sum(ts) / len(ts)
    out["adaptive_speedup_over_direct"] = out["direct_ms"] / out["adaptive_ms"]
    out["warp_speedup_over_direct"] = out["direct_ms"] / out["warp_ms"]
    out["note"] = ("each launch alone, L2 flushed before it, the host launch latency outside the events, "
                   "gradient zeroing included")
    return out


def time_preprocess(api, params, bufs, cam, opt, grads, sh_degree, flush, stream, reps: int) -> dict:
    """The two HBM-bound kernels of the step, gs_preprocess and gs_preprocess_bwd (one launch each),
    timed alone with L2 flushed before every launch (mean of `reps` launches), against their
    algorithmic bytes: the preprocess reads the geometry (40 B) of every Gaussian and the SH row and
    opacity logit of the visible ones, and writes the record, depth, radius and tile count (60 B) of
    every Gaussian; the backward reads every radius and, for the visible Gaussians, the parameters
    and the 48-byte 2D gradient, and writes every Gaussian's gradient row (zeros when culled)."""
    import torch
    peaks = load_json(PEAKS_PATH) or {}
    hbm = float(peaks.get("hbm_gbs", 6800.0))
    n = params["mean3d"].shape[0]
    sh4 = 3 * (sh_degree + 1) ** 2 * 4
    out = {}
    for name in ("preprocess", "preprocess_bwd"):
        ts = []
        for it in range(reps + 2):
            flush_l2(flush)
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            if name == "preprocess":
                api.gs_preprocess(params, cam, opt, out=bufs.proj)
            else:
                api.gs_preprocess_bwd(params, cam, opt, bufs.proj, bufs.grad2d, out=grads)
            e1.record(stream)
            torch.cuda.synchronize()
            if it >= 2:
                ts.append(e0.elapsed_time(e1))
        out[f"{name}_ms"] = sum(ts) / len(ts)
    vis = int((bufs.proj.radius > 0).sum().item())
    fwd_bytes = n * (40 + 60) + vis * (sh4 + 4)
    bwd_bytes = n * (4 + 44 + sh4) + vis * (40 + 48 + 4 + sh4)
    for name, b in (("preprocess", fwd_bytes), ("preprocess_bwd", bwd_bytes)):
        gbs = b / (out[f"{name}_ms"] / 1e3) / 1e9
        out[name] = {"algorithmic_bytes": b, "achieved_gbs": gbs, "frac_of_measured_hbm": gbs / hbm}
    out["visible"] = vis
    out["note"] = "each launch alone, L2 flushed before it, the host launch latency outside the events"
    return out


def config_block(cfg: int, dev, flush, stream, args, cpu: bool) -> dict:
    """The step of one configuration as one CUDA graph replay per step: ms per view, the raster
    kernels' times, duplicates per view and Mpix/s (5 timed replays, L2 flushed before each),
    and the oracle's rate on a window of the first view."""
    import torch
    import gs_scenes
    from differentiable_gaussian_splatting_gs_gb300 import api, step
    scene = gs_scenes.make_scene(cfg)
    names = ("mean3d", "log_scale", "quat", "opacity_logit", "sh")
    params = {k: torch.from_numpy(np.ascontiguousarray(getattr(scene, k))).to(dev) for k in names}
    grads = api.alloc_param_grads(params)
    cams = [api.make_camera(c) for c in scene.cameras]
    targets = [torch.from_numpy(t).to(dev) for t in scene.targets[:len(cams)]]
    opt = api.make_options(scene.sh_degree)
    bufs = step.StepBuffers(scene.n, dev)
    # capacity: the synchronising sort of every view, once
    cap = 0
    for c in cams:
        proj = api.gs_preprocess(params, c, opt, out=bufs.proj)
        cap = max(cap, api.gs_bin_and_sort(proj, c, opt, buffers=bufs.sort, want_keys=False).n_dup)
    ev = [((torch.cuda.Event(enable_timing=True, external=True), torch.cuda.Event(enable_timing=True, external=True)),
           (torch.cuda.Event(enable_timing=True, external=True), torch.cuda.Event(enable_timing=True, external=True)))
          for _ in cams]
    bufs2 = step.StepBuffers(scene.n, dev) if len(cams) > 1 else None  # views on two streams
    g = step.GraphedStep(params, cams, targets, opt, grads, bufs, cap + 1024, events=ev, buffers2=bufs2)
    for _ in range(3):
        g.replay()
    ms, fwd, bwd = [], [], []
    for _ in range(5):
        flush_l2(flush)
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        g.replay()
        e1.record(stream)
        torch.cuda.synchronize()
        ms.append(e0.elapsed_time(e1))
        fwd.append(sum(e[0][0].elapsed_time(e[0][1]) for e in ev) / len(cams))
        bwd.append(sum(e[1][0].elapsed_time(e[1][1]) for e in ev) / len(cams))
    views = len(cams)
    P = cams[0].width * cams[0].height
    m = sum(ms) / len(ms)
    out = {"workload": WORKLOADS[cfg], "views_per_step": views, "ms_per_view": m / views,
           "views_on_two_streams": bufs2 is not None,  # then fwd/bwd_ms include the other stream's overlap
           "mpix_per_s": P * views / (m / 1e3) / 1e6, "fwd_ms": sum(fwd) / len(fwd), "bwd_ms": sum(bwd) / len(bwd),
           "duplicates_per_view": int(g.n_dup.sum().item()) / views, "launches_per_step": g.launches}
    del g, bufs, bufs2, params, grads, targets
    if cpu:
        pix, dt, desc, cores = oracle_sample(scene, 0.25, 0.25)
        out["cpu_baseline"] = {"value": pix / dt / 1e6, "unit": "Mpix/s", "cores": cores, "kind": "oracle",
                               "sample": desc, "seconds": dt}
    return out


# ------------------------------------------------------------------------------------ reference arm

def run_reference(args, rank, world):
    if rank != 0:
        return
    import gs_scenes
    import oracle
    oracle.build()
    scene = gs_scenes.make_scene(CFG)
    frac = 0.25  # a quarter of the tiles in each direction: 1/16 of the pixels
    times, pix, desc = [], 0, ""
    for i in range(args.warmup + args.steps):
        pix, dt, desc, cores = oracle_sample(scene, frac, frac)
        if i >= args.warmup:
            times.append(dt)
    t = sum(times) / len(times)
    value = pix / t / 1e6
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": "Mpix/s", "n_gpus": args.gpus,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * t, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": WORKLOAD, "sample": desc},
            "cpu_baseline": {"value": value, "unit": "Mpix/s", "cores": os.cpu_count(), "kind": "oracle",
                             "sample": desc},
            "e2e": {"value": value, "unit": "Mpix/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


# ------------------------------------------------------------------------------------ our arm

def run_ours(args, rank, world, local_rank):
    import torch
    import torch.distributed as dist

    import gs_scenes
    import __graft_entry__
    from differentiable_gaussian_splatting_gs_gb300 import _abi, api, step

    __graft_entry__.build()
    torch.cuda.set_device(local_rank)
    dev = torch.device("cuda", local_rank)
    lib = _abi.load()

    scene = gs_scenes.make_scene(args.config)
    cam = scene.cameras[0]
    n_views = len(scene.cameras)
    P = cam.width * cam.height * n_views  # pixels per step (all views have the same size)
    names = ("mean3d", "log_scale", "quat", "opacity_logit", "sh")
    host = {k: torch.from_numpy(np.ascontiguousarray(getattr(scene, k))).pin_memory() for k in names}
    host_target = torch.from_numpy(np.stack(scene.targets[:n_views])).pin_memory()
    params = {k: host[k].to(dev) for k in names}
    target = host_target.to(dev)
    grads = api.alloc_param_grads(params)
    host_grads = {k: torch.empty_like(host[k]).pin_memory() for k in names}
    opt = api.make_options(scene.sh_degree, bwd_mode=args.mode, staging=args.staging,
                           adaptive_threshold=args.threshold)
    bufs = step.StepBuffers(scene.n, dev)
    flush = torch.empty(256 * 1024 * 1024 // 4, dtype=torch.float32, device=dev)
    stream = torch.cuda.current_stream(dev)

    cams = [api.make_camera(c) for c in scene.cameras]

    n_dup_dev = torch.zeros(n_views, dtype=torch.int64, device=dev)
    sort_sync = [True]  # the warm-up steps size the sort buffers with the synchronising call

    def one_step(ev_bwd=None, ev_fwd=None):
        """All views of one step; the views' parameter gradients are summed. ev_bwd / ev_fwd: one
        event pair per view around the backward / forward raster. After the warm-up the sort does
        not synchronise (the whole step is enqueued ahead of the GPU) and D lands in n_dup_dev."""
        n_dup = 0
        for v, c in enumerate(cams):
            proj = api.gs_preprocess(params, c, opt, out=bufs.proj)
            image, t_final, n_contrib, dl, ranges = bufs.image_buffers(c.width, c.height)
            if sort_sync[0]:
                b = api.gs_bin_and_sort(proj, c, opt, buffers=bufs.sort, ranges=ranges, want_keys=False)
                n_dup += b.n_dup
            else:
                b = api.gs_bin_and_sort_async(proj, c, opt, bufs.sort.capacity, buffers=bufs.sort, ranges=ranges,
                                              n_dup=n_dup_dev[v:v + 1])
            if ev_fwd is not None:
                ev_fwd[v][0].record(stream)
            api.gs_render_fwd(proj, b.vals, b.ranges, c, opt, out=(image, t_final, n_contrib))
            if ev_fwd is not None:
                ev_fwd[v][1].record(stream)
            if ev_bwd is not None:
                ev_bwd[v][0].record(stream)
            api.gs_render_bwd_sqerr(proj, b.vals, b.ranges, c, opt, image, target[v], t_final, n_contrib,
                                    grad2d=bufs.grad2d)
            if ev_bwd is not None:
                ev_bwd[v][1].record(stream)
            api.gs_preprocess_bwd(params, c, opt, proj, bufs.grad2d, out=grads, accumulate=v > 0)
        return n_dup

    def barrier():
        if world > 1:
            dist.barrier()

    for _ in range(max(args.warmup, 3)):
        n_dup = one_step()
    sort_sync[0] = args.sync_sort
    one_step()  # the step as timed, once more untimed
    torch.cuda.synchronize()
    assert api.gs_device_error() == 0

    # ---- the step as one CUDA graph: every kernel of the step with one host launch. The raster
    # kernels' events are captured in the graph as event record nodes (external events), so they
    # are timed inside each replay of the timed region.
    use_graph = not (args.no_graph or args.sync_sort)
    if use_graph:
        try:
            torch.cuda.Event(enable_timing=True, external=True)
        except TypeError:  # a torch without external events: the eager step is timed instead
            use_graph = False
    gstep = None
    if use_graph:
        def xev():
            return torch.cuda.Event(enable_timing=True, external=True)
        gev = [((xev(), xev()), (xev(), xev())) for _ in cams]
        bufs2 = step.StepBuffers(scene.n, dev) if n_views > 1 else None  # views on two streams
        gstep = step.GraphedStep(params, cams, [target[v] for v in range(n_views)], opt, grads, bufs,
                                 bufs.sort.capacity, events=gev, buffers2=bufs2)
        for _ in range(3):
            gstep.replay()
        torch.cuda.synchronize()
        assert api.gs_device_error() == 0

    # ---- device-resident timing: K steps, L2 flushed between steps (outside the events)
    step_ms, bwd_ms, fwd_ms = [], [], []
    launches0 = lib.gs_kernel_launches()
    barrier()
    torch.cuda.synchronize()
    with ClockSampler(local_rank) as clk:
        for _ in range(args.steps):
            flush_l2(flush)
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            if use_graph:
                ef, eb = [e[0] for e in gev], [e[1] for e in gev]
                e0.record(stream)
                gstep.replay()
                e1.record(stream)
            else:
                eb = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in cams]
                ef = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in cams]
                e0.record(stream)
                one_step(eb, ef)
                e1.record(stream)
            torch.cuda.synchronize()
            step_ms.append(e0.elapsed_time(e1))
            bwd_ms.append(sum(e[0].elapsed_time(e[1]) for e in eb) / n_views)  # per view
            fwd_ms.append(sum(e[0].elapsed_time(e[1]) for e in ef) / n_views)
    barrier()
    torch.cuda.synchronize()
    # kernels replayed from a graph are counted once at capture: per replay times the replays
    launches = gstep.launches * args.steps if use_graph else lib.gs_kernel_launches() - launches0
    assert api.gs_device_error() == 0
    if use_graph:
        n_dup = int(gstep.n_dup.sum())
    elif not args.sync_sort:
        n_dup = int(n_dup_dev.sum())
    launch_mode = (f"one CUDA graph per step ({gstep.launches} library kernels)" if use_graph else
                   "eager launches" + (", synchronising sort" if args.sync_sort else ", non-synchronising sort"))
    ms = reduce_max(sum(step_ms) / len(step_ms), world, dev)
    value = throughput_mpix(world, P, ms)

    # ---- end to end through the C ABI's host-buffer entry point (gs_train_step_host): every step
    # copies its parameters and target in from pinned host memory and its parameter gradients, loss
    # and D back, inside the timed region
    e2e = None
    if not args.no_e2e and n_views == 1:
        n_dup_e2e = int(gstep.n_dup.sum()) if use_graph else int(n_dup_dev.sum()) if not args.sync_sort else n_dup
        cap_e2e = max(1024, int(n_dup_e2e * 1.05) + 1024)
        NC = 3  # contexts (and streams) that take the steps in turn
        ctxs = [api.StepContext(scene.n, scene.sh_degree, cam.width, cam.height, cap_e2e) for _ in range(NC)]
        hin = [host] + [{k: torch.empty_like(v).pin_memory().copy_(v) for k, v in host.items()} for _ in range(NC - 1)]
        htg = [host_target[0]] + [host_target[0].clone().pin_memory() for _ in range(NC - 1)]
        hout = [host_grads] + [{k: torch.empty_like(v).pin_memory() for k, v in host.items()} for _ in range(NC - 1)]
        hloss = [torch.zeros(1).pin_memory() for _ in range(NC)]
        hdup = [torch.zeros(1, dtype=torch.int64).pin_memory() for _ in range(NC)]
        streams = [torch.cuda.Stream(dev) for _ in range(NC)]
        h2d = sum(t.numel() * t.element_size() for t in host.values()) + htg[0].numel() * 4
        d2h = sum(t.numel() * t.element_size() for t in host.values()) + 4 + 8

        def e2e_run(K, nctx):
            """K steps through gs_train_step_host, alternating over nctx contexts and streams; ms per step."""
            torch.cuda.synchronize()
            barrier()
            t0 = torch.cuda.Event(enable_timing=True)
            t0.record(streams[0])
            for s_ in streams[1:nctx]:
                s_.wait_event(t0)
            for kstep in range(K):
                b = kstep % nctx
                api.gs_train_step_host(ctxs[b], hin[b], htg[b], cam, opt, hout[b], hloss[b], hdup[b],
                                       stream=streams[b])
            ends = []
            for s_ in streams[:nctx]:
                e_ = torch.cuda.Event(enable_timing=True)
                e_.record(s_)
                ends.append(e_)
            torch.cuda.synchronize()
            barrier()
            return max(t0.elapsed_time(e_) for e_ in ends) / K

        K = max(6, args.steps)
        e2e_run(NC, NC)  # warm-up of every context
        serial = [e2e_run(K, 1) for _ in range(2)]
        runs = [e2e_run(K, NC) for _ in range(3)]
        assert api.gs_device_error() == 0
        assert int(hdup[0][0]) == n_dup_e2e, "the host-buffer step's D differs from the timed step's"
        em_serial = reduce_max(min(serial), world, dev)
        # the median of three timed pipelines (host memory and its link are shared with other devices
        # and processes; one run can be slowed by traffic that is not ours)
        em = reduce_max(statistics.median(runs), world, dev)
        e2e = {"value": throughput_mpix(world, P, em), "unit": "Mpix/s", "ms_per_step": em,
               "h2d_bytes_per_step": int(h2d), "d2h_bytes_per_step": int(d2h),
               "call": "gs_train_step_host (C ABI, host buffers in and out, one cudaMemcpyAsync per array)",
               "pipeline": f"{NC} step contexts on {NC} streams in turn: a step's copies in, compute and copies out "
                           "overlap its neighbours'",
               "serial_ms_per_step": em_serial, "pipelined_runs_ms": runs}
        # the host link alone: what the copies of one step take at the link's own rate (copy engines,
        # pinned memory, both directions at once, as in the pipeline), against the step's period
        link = host_link_gbs(host["sh"], torch.empty_like(grads["sh"]), stream)
        link_ms = max(h2d, d2h) / (link["both_gbs_each"] * 1e6)
        e2e["host_link"] = dict(link, copy_ms_per_step=link_ms, frac=link_ms / em)
        for c_ in ctxs:
            c_.close()
    assert api.gs_device_error() == 0

    # ---- the update phase after the step (not part of the fwd+bwd metric): sparse Adam over the
    # Gaussians the view made visible, timed alone with L2 flushed before each launch
    extras = {}
    if not args.no_extras and use_graph:
        # the same step with eager launches (non-synchronising sort), for comparison with the graph
        q_ms = []
        for _ in range(max(3, args.steps // 2)):
            flush_l2(flush)
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            one_step()
            e1.record(stream)
            torch.cuda.synchronize()
            q_ms.append(e0.elapsed_time(e1))
        qm = sum(q_ms) / len(q_ms)
        extras["eager_step"] = {"ms_per_step": qm, "mpix_per_s": P / (qm / 1e3) / 1e6}
        assert api.gs_device_error() == 0
    if not args.no_extras:
        # the backward raster in each accumulation mode on this step's own inputs, each launch timed
        # alone with L2 flushed before it (the pages' comparison: warp-level reduction against direct
        # per-thread atomics, DISTWAR Abstract)
        one_step()
        torch.cuda.synchronize()
        extras["bwd_modes"] = time_bwd_modes(api, bufs, cams[-1], target[n_views - 1], scene.sh_degree, flush,
                                             stream, max(5, args.steps // 2))
        assert api.gs_device_error() == 0
        extras["preprocess"] = time_preprocess(api, params, bufs, cams[-1], opt, grads, scene.sh_degree, flush,
                                               stream, max(5, args.steps // 2))
        assert api.gs_device_error() == 0
        exp_avg = {k: torch.zeros_like(params[k]) for k in names}
        exp_avg_sq = {k: torch.zeros_like(params[k]) for k in names}
        radius = bufs.proj.radius
        n_vis = int((radius > 0).sum().item())
        floats = sum(params[k][0].numel() for k in names)
        a_ms = []
        for t in range(1, 4 + max(3, args.steps // 2)):
            flush_l2(flush)
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            api.gs_adam_step(params, grads, exp_avg, exp_avg_sq, radius,
                             api.make_adam_options(gs_scenes.ADAM_LR, t, scene.sh_degree))
            e1.record(stream)
            torch.cuda.synchronize()
            if t > 3:
                a_ms.append(e0.elapsed_time(e1))
        am = sum(a_ms) / len(a_ms)
        a_bytes = n_vis * floats * 4 * 7 + scene.n * 4  # p, m, v read + written, g read; radius
        peaks = load_json(PEAKS_PATH) or {}
        hbm = float(peaks.get("hbm_gbs", 6800.0))
        extras["sparse_adam"] = {"ms": am, "visible": n_vis, "algorithmic_bytes": a_bytes,
                                 "achieved_gbs": a_bytes / (am / 1e3) / 1e9,
                                 "frac_of_measured_hbm": a_bytes / (am / 1e3) / 1e9 / hbm}
        # post-backward statistics: densification accumulators and per-Gaussian gradient magnitudes
        acc = torch.zeros(scene.n, device=dev)
        cnt = torch.zeros(scene.n, dtype=torch.int32, device=dev)
        mrad = torch.zeros(scene.n, dtype=torch.int32, device=dev)
        gmag = torch.empty(scene.n, device=dev)
        s_ms = []
        for it in range(4 + max(3, args.steps // 2)):
            flush_l2(flush)
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            api.gs_densify_stats(bufs.proj, bufs.grad2d, cam.width, cam.height, acc, cnt, mrad,
                                 param_grads=grads, grad_mag=gmag, sh_degree=scene.sh_degree)
            e1.record(stream)
            torch.cuda.synchronize()
            if it > 3:
                s_ms.append(e0.elapsed_time(e1))
        sm_ = sum(s_ms) / len(s_ms)
        s_bytes = scene.n * 8 + n_vis * (32 + 12 + floats * 4)  # radius + magnitude; grad2d sector, stats, grads
        extras["densify_stats"] = {"ms": sm_, "algorithmic_bytes": s_bytes, "achieved_gbs": s_bytes / (sm_ / 1e3) / 1e9,
                                   "frac_of_measured_hbm": s_bytes / (sm_ / 1e3) / 1e9 / hbm}
        # the same statistics emitted by the preprocess backward itself, against the plain backward
        pb_ms = {False: [], True: []}
        for it in range(4 + max(3, args.steps // 2)):
            for fused in (False, True):
                flush_l2(flush)
                e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                e0.record(stream)
                if fused:
                    api.gs_preprocess_bwd_stats(params, cams[n_views - 1], opt, bufs.proj, bufs.grad2d, acc, cnt,
                                                mrad, grad_mag=gmag, out=grads)
                else:
                    api.gs_preprocess_bwd(params, cams[n_views - 1], opt, bufs.proj, bufs.grad2d, out=grads)
                e1.record(stream)
                torch.cuda.synchronize()
                if it > 3:
                    pb_ms[fused].append(e0.elapsed_time(e1))
        extras["densify_stats"]["fused_into_preprocess_bwd"] = {
            "preprocess_bwd_ms": sum(pb_ms[False]) / len(pb_ms[False]),
            "preprocess_bwd_stats_ms": sum(pb_ms[True]) / len(pb_ms[True])}
        # image loss L1 + D-SSIM and dL/dimage of the rendered view
        image = bufs.image_buffers(cam.width, cam.height)[0]
        lws = torch.empty(int(lib.gs_loss_workspace_bytes(cam.width, cam.height)), dtype=torch.uint8, device=dev)
        lout = (torch.empty(1, device=dev), torch.empty_like(image))
        l_ms = []
        for it in range(4 + max(3, args.steps // 2)):
            flush_l2(flush)
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            api.gs_loss_l1_dssim(image, target[n_views - 1], 0.2, workspace=lws, out=lout)
            e1.record(stream)
            torch.cuda.synchronize()
            if it > 3:
                l_ms.append(e0.elapsed_time(e1))
        lm = sum(l_ms) / len(l_ms)
        l_bytes = cam.width * cam.height * 3 * 4 * (2 + 3 + 3 + 2 + 1)  # pass 1: x, y in, 3 maps out; pass 2: 3 maps, x, y in, dL out
        extras["loss_l1_dssim"] = {"ms": lm, "algorithmic_bytes": l_bytes, "achieved_gbs": l_bytes / (lm / 1e3) / 1e9,
                                   "frac_of_measured_hbm": l_bytes / (lm / 1e3) / 1e9 / hbm}
        # the surfel (2D Gaussian splatting) step on the same parameters and view
        rec2d = torch.empty((scene.n, 16), dtype=torch.float32, device=dev)
        g2d = torch.empty((scene.n, 16), dtype=torch.float32, device=dev)
        c0 = cams[0]

        def step2d(ev=None):
            mark = (lambda i: ev[i].record(stream)) if ev else (lambda i: None)
            proj2, _ = api.gs_preprocess2d(params, c0, opt, out=bufs.proj, rec2d=rec2d)
            mark(0)
            image2, t2, nc2, dl2, ranges2 = bufs.image_buffers(c0.width, c0.height)
            b2 = api.gs_bin_and_sort(proj2, c0, opt, buffers=bufs.sort, ranges=ranges2, want_keys=False)
            mark(1)
            api.gs_render2d_fwd(rec2d, b2.vals, b2.ranges, c0, opt, out=(image2, t2, nc2))
            mark(2)
            torch.sub(image2, target[0], out=dl2)
            mark(3)
            api.gs_render2d_bwd(rec2d, b2.vals, b2.ranges, c0, opt, dl2, t2, nc2, grad2d=g2d)
            mark(4)
            api.gs_preprocess2d_bwd(params, c0, opt, proj2, g2d, out=grads)
            return b2.n_dup
        for _ in range(3):
            step2d()
        s_ms2, parts = [], []
        for _ in range(max(3, args.steps // 2)):
            flush_l2(flush)
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            ev = [torch.cuda.Event(enable_timing=True) for _ in range(5)]
            e0.record(stream)
            d2 = step2d(ev)
            e1.record(stream)
            torch.cuda.synchronize()
            s_ms2.append(e0.elapsed_time(e1))
            marks = [e0] + ev + [e1]
            parts.append([marks[i].elapsed_time(marks[i + 1]) for i in range(6)])
        m2 = sum(s_ms2) / len(s_ms2)
        pm = [sum(p[i] for p in parts) / len(parts) for i in range(6)]
        # the surfel step as one CUDA graph (non-synchronising sort), on the same buffers
        g2step = step.GraphedStep(params, [c0], [target[0]], opt, grads, bufs, bufs.sort.capacity, surfels=True)
        for _ in range(3):
            g2step.replay()
        q_ms = []
        for _ in range(max(3, args.steps // 2)):
            flush_l2(flush)
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            g2step.replay()
            e1.record(stream)
            torch.cuda.synchronize()
            q_ms.append(e0.elapsed_time(e1))
        gm2 = sum(q_ms) / len(q_ms)
        extras["surfel_step"] = {"ms_per_view": m2, "mpix_per_s": c0.width * c0.height / (m2 / 1e3) / 1e6,
                                 "graph_ms_per_view": gm2,
                                 "graph_mpix_per_s": c0.width * c0.height / (gm2 / 1e3) / 1e6,
                                 "duplicates": int(d2),
                                 "stage_ms": dict(zip(["preprocess", "bin_and_sort", "render_fwd", "dl_dimage",
                                                       "render_bwd", "preprocess_bwd"], pm))}
        assert api.gs_device_error() == 0
    if not args.no_extras and use_graph and world == 1 and args.config == CFG:
        # every configuration measured the same way in this run (fields of the metric per config),
        # with the oracle's CPU rate on a window of each view beside it
        del g2step
        extras["configs"] = {}
        for c in sorted(WORKLOADS):
            extras["configs"][str(c)] = config_block(c, dev, flush, stream, args, cpu=not args.no_cpu_baseline)
            torch.cuda.empty_cache()
        assert api.gs_device_error() == 0

    # ---- roofline of the dominant kernel (the backward)
    peaks = load_json(PEAKS_PATH) or {}
    counts = json_block(COUNTS_PATH) or {}
    clocks = clk.summary()
    bwd_avg_ms = sum(bwd_ms) / len(bwd_ms)
    roof = None
    if "pairs_replayed_bwd" in counts and args.config == CFG:
        roof = backward_roofline(counts, peaks, bwd_avg_ms, dev, args.mode)

    line = {"metric": METRIC, "value": value, "unit": "Mpix/s", "n_gpus": world, "steps": args.steps,
            "warmup": max(args.warmup, 3), "ms_per_step": ms, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f32", "data": "synthetic",
            "config": {"workload": WORKLOADS[args.config], "n_gaussians": scene.n, "width": cam.width,
                       "height": cam.height, "views_per_step": n_views, "duplicates": int(n_dup), "bwd_mode": args.mode,
                       "l2": "flushed between timed steps (256 MB write and a 0.1 ms device wait, both outside the events)",
                       "parallelism": f"replicas x{world}", "launch": launch_mode},
            "roofline": roof, "e2e": e2e, "gpu_launches": int(launches), "clocks": clocks,
            "bwd_ms": bwd_avg_ms, "fwd_ms": sum(fwd_ms) / len(fwd_ms), "ms_per_view": ms / n_views, "step_ms_min": min(step_ms), "extras": extras}
    if rank == 0 and world == 1 and not args.no_cpu_baseline and n_views == 1:
        # the oracle's whole step on the whole view, repeated until about 10 s of CPU time
        runs = []
        while sum(runs) < 10.0 and len(runs) < 5:
            pix, dt, desc, cores = oracle_sample(scene, 1.0, 1.0)
            runs.append(dt)
        dt = sum(runs) / len(runs)
        line["cpu_baseline"] = {"value": pix / dt / 1e6, "unit": "Mpix/s", "cores": cores, "kind": "oracle",
                                "sample": f"{desc}; mean of {len(runs)} runs", "seconds": dt}
    if rank == 0:
        print(json.dumps(line), flush=True)


def main():
    args = parse_args()
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local_rank = int(os.environ.get("LOCAL_RANK", "0"))
    if args.impl == "reference":
        # the CPU oracle runs on rank 0 only; other ranks have no work
        if rank == 0:
            run_reference(args, rank, world)
        return
    if world > 1:
        import torch.distributed as dist
        import torch
        torch.cuda.set_device(local_rank)
        dist.init_process_group("nccl")
    try:
        run_ours(args, rank, world, local_rank)
    finally:
        if world > 1:
            import torch.distributed as dist
            dist.destroy_process_group()


if __name__ == "__main__":
    main()
