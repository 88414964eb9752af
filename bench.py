#!/usr/bin/env python
"""Benchmark of the tile-based differentiable sphere renderer on one GB300.

Metric: forward + backward frames/s (and Msphere-pixel/s = hit pairs / time)
on the 1,000,000-sphere 1024x1024 scene (3 channels, n_track 5, camera R/t/K
gradients) -- the scale of the Pulsar paper's 1M-sphere timings (Sec. 1,
Table 2).  One step = project -> bin -> forward -> backward (all kernels of
the path) over one frame, replayed from a CUDA graph, inputs resident in HBM,
L2 flushed between steps by a 256 MB write.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl gb300|reference]

With N > 1 (torchrun) every rank renders its own frame: replicas, weak
scaling, no collective on the data path.  `--impl reference` times the CPU
oracle (fp64, all host cores) on a bounded sample of the same frame.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

WORKLOAD = "headline: 1,000,000 spheres, 1024x1024, 3 channels, n_track 5, R/t/K gradients"
WORKLOADS = {
    "headline": WORKLOAD,
    "headline_ortho": "headline sizes, orthographic camera: 1,000,000 spheres, 1024x1024, "
                      "3 channels, n_track 5, R/t/K gradients",
    "neural": "neural: 1,000,000 spheres, 1024x1024, 16 channels, n_track 8, R/t/K gradients",
    "driving": "driving rig: 2,000,000 spheres, six 1920x1080 cameras in one batched launch, "
               "3 channels, n_track 5, R/t/K gradients; value in camera frames/s",
    "neural_shaded": "neural pipeline: the neural scene (1,000,000 spheres, 1024x1024, 16 "
                     "channels, n_track 8) rendered, shaded to RGB by the per-pixel MLP "
                     "(19-64-64-3, bf16 tensor cores), MLP backward, render backward fed with "
                     "dL/dF; gradients of spheres, camera and MLP weights",
}
METRIC = "fwd+bwd frames/s at 1M spheres 1024^2"
UNIT = "frames/s"
KERNELS_PER_STEP = 9   # project, tile_scan, emit, tile_sort, tile_sort_long, forward, backward,
                       # finalize, camera_reduce
SHADE_KERNELS = 5      # weight pack + shade forward, weight pack + shade backward + reduce


def args_parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=50)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", default="gb300", choices=["gb300", "reference"])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-scenes", action="store_true",
                    help="headline only: skip timing the neural and driving configurations")
    ap.add_argument("--cpu-seconds", type=float, default=12.0,
                    help="target CPU time of the oracle sample")
    ap.add_argument("--scene", default="headline", choices=sorted(WORKLOADS),
                    help="workload (the default is the headline configuration)")
    ap.add_argument("--cams", type=int, default=0,
                    help="driving rig: render only its first CAMS cameras (0: all six)")
    ap.add_argument("--frames-only", type=int, default=0,
                    help="render and differentiate this many frames eagerly, print nothing "
                         "(a short fixed launch sequence for profilers)")
    return ap.parse_args()


def dist_env():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def max_over_ranks(value: float, dist, device) -> float:
    """The largest of every rank's value (the slowest replica's time); the
    value itself for a single process (dist None)."""
    if not dist:
        return value
    import torch
    t = torch.tensor([value], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_rate(world: int, units_per_rank_step: int, steps: int, total_ms: float) -> float:
    """Whole-job throughput: the units all replicas processed over the slowest
    replica's time (replicas render independent frames; no data-path exchange)."""
    return world * units_per_rank_step * steps / (total_ms * 1e-3)


# ------------------------------------------------------------------ clocks --
class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, device_index: int):
        self.dev = device_index
        self.p = None

    def start(self):
        try:
            self.p = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "50", "-i", str(self.dev)], stdout=subprocess.PIPE,
                stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.p = None

    def stop(self):
        if self.p is None:
            return None
        self.p.terminate()
        try:
            out, _ = self.p.communicate(timeout=5)
        except subprocess.TimeoutExpired:
            self.p.kill()
            out, _ = self.p.communicate()
        sm, mx, reasons = [], 0.0, set()
        names = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")
        for line in out.splitlines():
            f = [x.strip() for x in line.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                mx = max(mx, float(f[2]))
            except ValueError:
                continue
            for n, v in zip(names, f[5:9]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        if not sm:
            return None
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": mx, "reasons": sorted(reasons),
                "samples": len(sm)}


# -------------------------------------------------------------- roofline --
def measured_peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            return json.load(f), "measured"
    except OSError:
        return {"hbm_gbs": 6800.0, "sm_max_mhz": 2070.0}, "fallback"


# FP32 peak of the ALU-bound kernels: SMs (read from the device) x 128 FP32
# lanes x 2 flops (FMA) at the maximum SM clock of MEASURED_PEAKS (2070 MHz).
FP32_LANES = 128


def fp32_peak_tflops(peaks, sms: int) -> float:
    return sms * FP32_LANES * 2 * float(peaks.get("sm_max_mhz", 2070.0)) * 1e6 / 1e12


def algorithmic_bytes(stage, N, M, P, C, T):
    """Compulsory bytes of one launch of each stage: every array moved once,
    sphere records gathered once per sphere-tile pair in the forward and once
    per sphere in the backward (the per-unit figures of the hot-path table)."""
    if stage == "project":
        return 20 * N + 44 * N
    if stage == "bin":
        return 8 * N + 12 * N + 12 * M + 24 * M + 8 * M
    if stage == "forward":
        return 4 * M + (32 + 4 * C) * M + 4 * C * P + (8 + 4 * T) * P
    if stage == "backward":
        return (8 * C * P + (8 + 4 * T) * P + (32 + 4 * C) * N + (20 + 4 * C) * N + 12 * N
                + 24 * N + 12 * N)
    raise KeyError(stage)


def algorithmic_flops(stage, N, M, P, C, T, H, Ht):
    """FP32 work of the method (FMA = 2): the cooperative candidate test of
    every tile pair at every pixel of its 16x16 tile (~14 flops), the blend of
    every hit (12 + 2C), the tracked-hit gradient (70 + 6C), the projection
    (~100 per sphere)."""
    if stage == "project":
        return 100 * N
    if stage == "forward":
        return 14 * M * 256 + (12 + 2 * C) * H
    if stage == "backward":
        return (70 + 6 * C) * Ht
    return 0


# Shading MLP per pixel: compulsory HBM bytes (features 64 B in, rgb 12 B out;
# backward: features and dL/drgb in, dL/dF 64 B out) and tensor-core flops
# (forward 2 x (19*64 + 64*64 + 64*3); backward: the two hidden layers again,
# W3^T, W2^T, W1^T[:16] products, and the weight and bias gradients).
SHADE_BYTES_PER_PIXEL = {"shade_forward": 64 + 12, "shade_backward": 64 + 12 + 64}
SHADE_FLOPS_PER_PIXEL = {"shade_forward": 2 * (19 * 64 + 64 * 64 + 64 * 3),
                         "shade_backward": 2 * (19 * 64 + 64 * 64 + 3 * 64 + 64 * 64 + 64 * 16
                                                + 64 * 20 + 64 * 65 + 3 * 65)}


def traffic_from_profile(kernel: str, source: str, workload: str):
    """DRAM bytes per launch recorded by the committed ncu summary of `kernel`,
    if it was taken on the current source; else None."""
    path = os.path.join(ROOT, "profiles", f"{kernel}_{workload}.txt")
    src = os.path.join(ROOT, "splat_rendering_gb300", "csrc")
    try:
        with open(path) as f:
            kv = dict(l.split(":", 1) for l in f.read().splitlines() if ":" in l)
        h = hashlib.sha256()
        for name in ("pulsar_internal.cuh", source):
            with open(os.path.join(src, name), "rb") as g:
                h.update(g.read())
        if kv.get("source_sha256", "").strip() != h.hexdigest():
            return None
        return float(kv["dram_bytes_per_launch"])
    except (OSError, KeyError, ValueError):
        return None


# ------------------------------------------------------------- reference --
def oracle_sample(scene, target_s: float, rows: int | None = None, shade=None):
    """Time the CPU oracle on a band of rows of the frame (forward + backward;
    with shade = (mlp weights, dL/drgb): forward, the shading MLP forward and
    backward, and the render backward fed with its dL/dF).  With rows=None
    the band grows until it takes about target_s, and whole frames are
    repeated when one frame is quicker.  Returns (frames/s extrapolated by the
    pixel fraction, rows, seconds timed, cores, frames repeated)."""
    import dataclasses

    import numpy as np
    import oracle
    from oracle import mlp
    cam = scene.cameras[0]
    fixed = rows is not None
    rows = rows or 16

    def run_band():
        win = (0, 0, cam.width, rows)
        G = np.zeros_like(scene.grad_images[0])
        if shade is None:
            G[:rows] = scene.grad_images[0][:rows]
        else:
            F = oracle.render(scene.pos, scene.radius, scene.opacity, scene.features, cam,
                              scene.params, scene.bg, window=win)["image"]
            band = dataclasses.replace(cam, height=rows)
            g = mlp.backward(F.reshape(-1, 16), band, shade[0], shade[1][:rows].reshape(-1, 3))
            G[:rows] = g["grad_features"].reshape(rows, cam.width, 16)
        oracle.render(scene.pos, scene.radius, scene.opacity, scene.features, cam, scene.params,
                      scene.bg, grad_image=G, window=win)

    while True:
        t0 = time.perf_counter()
        run_band()
        dt = time.perf_counter() - t0
        if fixed or dt >= 0.5 * target_s or rows >= cam.height:
            break
        rows = min(cam.height, max(rows * 2, int(rows * 0.6 * target_s / max(dt, 1e-3))))
    frac = rows / cam.height
    reps = 1
    if not fixed and rows >= cam.height and dt < 0.5 * target_s:
        # the whole frame is quicker than the target: time whole frames back to back
        reps = min(50, max(1, int(0.6 * target_s / max(dt, 1e-3))))
        t0 = time.perf_counter()
        for _ in range(reps):
            run_band()
        dt = (time.perf_counter() - t0) / reps
    return frac / dt, rows, dt * reps, oracle.num_threads(), reps


def run_reference(a):
    world, rank, _ = dist_env()
    if rank != 0:
        return
    from splat_rendering_gb300 import scenes
    scene = scenes.headline()
    vals = []
    per_step = max(1.0, a.cpu_seconds / max(1, a.steps))
    rows = None
    for i in range(a.warmup + a.steps):
        v, rows, dt, cores, _ = oracle_sample(scene, per_step, rows)
        if i >= a.warmup:
            vals.append(v)
    value = statistics.median(vals)
    sample = (f"oracle fp64 fwd+bwd on rows [0,{rows}) x 1024 of the headline frame, "
              f"scaled by the pixel fraction {rows}/1024")
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": UNIT,
            "n_gpus": world, "steps": a.steps, "warmup": a.warmup,
            "ms_per_step": 1e3 / value, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": WORKLOAD, "parallelism": "replicas"},
            "cpu_baseline": {"value": value, "unit": UNIT, "cores": cores, "kind": "oracle",
                             "sample": sample},
            "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


# ----------------------------------------------------------------- gb300 --
class Workload:
    """One configuration on one device: inputs resident in HBM, a context sized
    for it, and one step (project -> bin -> forward [-> shading] -> backward)."""

    def __init__(self, name, dev, local, cams=0):
        import numpy as np
        import torch

        from splat_rendering_gb300 import pulsar as pl
        from splat_rendering_gb300 import scenes
        self.name, self.dev, self.pl = name, dev, pl
        self.shaded = name == "neural_shaded"
        scene = scenes.make("neural" if self.shaded else name)
        self.scene = scene
        # the driving rig renders its six cameras as one batch; the others one camera
        cams = scene.cameras[:cams or None] if name == "driving" else scene.cameras[:1]
        self.cams, self.K = cams, len(cams)
        K = self.K
        cam, prm = cams[0], scene.params
        self.cam, self.prm = cam, prm
        self.N, self.C, self.T = scene.n, prm.channels, prm.n_track
        self.P = cam.width * cam.height * K

        def dev_t(x):
            return torch.from_numpy(np.ascontiguousarray(x)).to(dev)

        self.dev_t = dev_t
        self.pos, self.rad, self.opa, self.feat = (dev_t(scene.pos), dev_t(scene.radius),
                                                   dev_t(scene.opacity), dev_t(scene.features))
        self.G_host = np.stack(scene.grad_images[:K]) if K > 1 else scene.grad_images[0]
        self.bg, self.G = dev_t(scene.bg), dev_t(self.G_host)
        self.c_cam = [pl.camera(c) for c in cams] if K > 1 else pl.camera(cam)
        self.c_prm = pl.params(prm)
        N, C = self.N, self.C
        self.image = torch.empty(((K,) if K > 1 else ()) + (cam.height, cam.width, C), device=dev)
        self.grads = {"pos": torch.empty((N, 3), device=dev), "radius": torch.empty(N, device=dev),
                      "opacity": torch.empty(N, device=dev),
                      "features": torch.empty((N, C), device=dev),
                      "cam": torch.empty(((K,) if K > 1 else ()) + (16,), device=dev)}
        self.cap = 4 * N
        self.local = local
        self.r = self._renderer(self.cap)
        if self.shaded:
            # per-pixel MLP shading: rgb = MLP(F); dL/drgb seeded; dL/dF feeds the render backward
            self.mlp_host = scenes.shading_mlp(5)
            self.drgb_host = scenes.shading_grad(7, cam.height, cam.width)
            self.mlp_w, self.drgb = dev_t(self.mlp_host), dev_t(self.drgb_host)
            self.rgb = torch.empty((cam.height, cam.width, 3), device=dev)
            self.gF = torch.empty_like(self.image)
            self.grads["mlp"] = torch.empty_like(self.mlp_w)

    def _renderer(self, cap):
        return self.pl.Renderer(max_spheres=self.N, max_pairs=cap, max_width=self.cam.width,
                                max_height=self.cam.height, max_channels=self.C,
                                max_track=self.T, device=self.local, max_cams=self.K)

    def step(self):
        r = self.r
        r.render(self.pos, self.rad, self.opa, self.feat, self.c_cam, self.c_prm, self.bg,
                 image=self.image)
        if self.shaded:
            r.shade(self.image, self.mlp_w, self.rgb)
            r.shade_backward(self.image, self.mlp_w, self.drgb, self.gF, self.grads["mlp"])
            r.backward(self.gF, out=self.grads)
        else:
            r.backward(self.G, out=self.grads)

    def first_frame(self):
        """Render once; grow the pair capacity if needed.  Sets M, H, Ht."""
        import numpy as np
        import torch
        pl = self.pl
        self.step()
        code, M, H = self.r.status(raise_on_error=False)
        if code == pl.ERR_CAPACITY:
            self.r.close()
            self.r = self._renderer(2 * M)
            self.step()
            code, M, H = self.r.status()
        assert code == 0, pl.strerror(code)
        ids = torch.from_numpy(self.r.debug("ids").view(np.int32))
        self.M, self.H, self.Ht = M, H, int((ids >= 0).sum())

    def graph(self):
        import torch
        s = torch.cuda.Stream(device=self.dev)
        s.wait_stream(torch.cuda.current_stream())
        with torch.cuda.stream(s):
            for _ in range(2):
                self.step()
        torch.cuda.current_stream().wait_stream(s)
        torch.cuda.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            self.step()
        torch.cuda.synchronize()
        return g

    def stages(self):
        return ("project", "bin", "forward") + (("shade_forward", "shade_backward")
                                                if self.shaded else ()) + ("backward",)

    def breakdown(self, steps, flush):
        """Per-stage device times: the same kernels eagerly, CUDA events between
        the ABI calls on the stream they launch on, L2 flushed before each step."""
        import torch
        pl, r, stages = self.pl, self.r, self.stages()
        per = {k: [] for k in stages}
        for _ in range(steps):
            flush.zero_()
            ev = [torch.cuda.Event(enable_timing=True) for _ in range(len(stages) + 1)]
            ev[0].record()
            if self.K > 1:
                pl.project_cams(r.ctx, self.pos, self.rad, self.opa, self.N, self.c_cam,
                                self.c_prm)
            else:
                pl.project(r.ctx, self.pos, self.rad, self.opa, self.N, self.c_cam, self.c_prm)
            ev[1].record()
            pl.bin(r.ctx)
            ev[2].record()
            pl.forward(r.ctx, self.feat, self.bg, self.image)
            ev[3].record()
            G_in = self.G
            if self.shaded:
                pl.shade_forward(r.ctx, self.image, self.mlp_w, self.rgb)
                ev[4].record()
                pl.shade_backward(r.ctx, self.image, self.mlp_w, self.drgb, self.gF,
                                  self.grads["mlp"])
                ev[5].record()
                G_in = self.gF
            g = self.grads
            pl.backward(r.ctx, self.feat, self.bg, self.image, G_in, g["pos"], g["radius"],
                        g["opacity"], g["features"], g["cam"])
            ev[-1].record()
            torch.cuda.synchronize()
            for i, k in enumerate(stages):
                per[k].append(ev[i].elapsed_time(ev[i + 1]))
        return {k: statistics.median(v) for k, v in per.items()}

    def rooflines(self, breakdown, step_ms, peaks, peak_src, sms):
        """Forward-kernel roofline and the whole path's, from the algorithmic
        byte and flop counts of each stage."""
        N, M, P, C, T, H, Ht = self.N, self.M, self.P, self.C, self.T, self.H, self.Ht
        hbm = float(peaks["hbm_gbs"])
        fp32 = fp32_peak_tflops(peaks, sms)
        clk = float(peaks.get("sm_max_mhz", 2070.0))
        fwd_flops = algorithmic_flops("forward", N, M, P, C, T, H, Ht)
        fwd_bytes = algorithmic_bytes("forward", N, M, P, C, T)
        fwd_s = breakdown["forward"] * 1e-3
        achieved = fwd_flops / fwd_s / 1e12
        roofline = {"bound": "alu", "kernel": "k_forward", "achieved": achieved, "peak": fp32,
                    "unit": "TFLOP/s", "frac": achieved / fp32,
                    "traffic": (traffic_from_profile("k_forward", "forward.cu", "headline")
                                if self.name == "headline" else None),
                    "algorithmic_flops": fwd_flops, "algorithmic_bytes": fwd_bytes,
                    "hbm_frac": fwd_bytes / fwd_s / 1e9 / hbm,
                    # secondary ceiling: two MUFU operations (exp2, rsqrt) per hit at
                    # 16 per SM and clock
                    "mufu_time_us": 2 * H / (sms * 16 * clk * 1e6) * 1e6,
                    "peak_source": f"FP32: {sms} SMs (read from the device) x {FP32_LANES} "
                                   f"lanes x 2 x {clk} MHz ({peak_src} clock); "
                                   f"HBM: {peak_src} hbm_gbs {hbm}"}
        render_stages = ("project", "bin", "forward", "backward")
        path_bytes = sum(algorithmic_bytes(k, N, M, P, C, T) for k in render_stages)
        path_flops = sum(algorithmic_flops(k, N, M, P, C, T, H, Ht) for k in render_stages)
        shade_roof = None
        if self.shaded:
            bf16 = float(peaks.get("bf16_tflops_sustained", 1700.0))   # inside a long step
            shade_roof = {}
            for k in ("shade_forward", "shade_backward"):
                b, fl = SHADE_BYTES_PER_PIXEL[k] * P, SHADE_FLOPS_PER_PIXEL[k] * P
                t_s = breakdown[k] * 1e-3
                shade_roof[k] = {"bound": "hbm", "achieved": b / t_s / 1e9, "peak": hbm,
                                 "unit": "GB/s", "frac": b / t_s / 1e9 / hbm,
                                 "algorithmic_bytes": b, "tensor_flops": fl,
                                 "tensor_frac": fl / t_s / 1e12 / bf16}
                path_bytes += b
        path_time = max(path_bytes / (hbm * 1e9), path_flops / (fp32 * 1e12))
        path = {"algorithmic_bytes": path_bytes, "algorithmic_flops": path_flops,
                "hbm_time_ms": path_bytes / (hbm * 1e9) * 1e3,
                "fp32_time_ms": path_flops / (fp32 * 1e12) * 1e3,
                "frac": path_time * 1e3 / step_ms}
        return roofline, path, shade_roof

    def close(self):
        self.r.close()


def time_graph(graph, steps, flush):
    """Per-step device times of graph replays, L2 flushed before each (outside
    the events)."""
    import torch
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
           for _ in range(steps)]
    torch.cuda.synchronize()
    for e0, e1 in evs:
        flush.zero_()
        e0.record()
        graph.replay()
        e1.record()
    torch.cuda.synchronize()
    return [e0.elapsed_time(e1) for e0, e1 in evs]


def side_scene(name, dev, local, steps, warmup, flush, peaks, peak_src, sms):
    """A further configuration timed the same way as the headline (graph replay
    of one step, L2 flushed between steps), for the run's record."""
    import numpy as np
    wl = Workload(name, dev, local)
    wl.first_frame()
    g = wl.graph()
    for _ in range(warmup):
        flush.zero_()
        g.replay()
    step_ms = time_graph(g, steps, flush)
    ms = statistics.median(step_ms)
    bd = wl.breakdown(max(3, steps // 2), flush)
    roof, path, shade = wl.rooflines(bd, ms, peaks, peak_src, sms)
    out = {"workload": WORKLOADS[name], "steps": steps, "ms_per_step": ms,
           "value": wl.K / (ms * 1e-3), "unit": UNIT if wl.K == 1 else "camera frames/s",
           "step_ms_quantiles": {q: float(np.quantile(step_ms, v)) for q, v in
                                 (("p10", 0.1), ("p90", 0.9))},
           "breakdown_ms": bd, "path_roofline": path,
           "forward_roofline": {k: roof[k] for k in ("achieved", "peak", "unit", "frac",
                                                      "hbm_frac")},
           "pairs_per_frame": wl.M, "hits_per_frame": wl.H, "tracked_hits_per_frame": wl.Ht}
    if shade:
        out["shade_roofline"] = shade
    del g
    wl.close()
    return out


def run_gb300(a):
    import numpy as np
    import torch

    from splat_rendering_gb300 import build as pbuild
    from splat_rendering_gb300 import pulsar as pl

    world, rank, local = dist_env()
    torch.cuda.set_device(local)
    dist = None
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl")
    pbuild.build()
    pl.load()
    dev = torch.device("cuda", local)
    sms = torch.cuda.get_device_properties(dev).multi_processor_count

    wl = Workload(a.scene, dev, local, a.cams)
    if a.frames_only:
        for _ in range(a.frames_only):
            wl.step()
        torch.cuda.synchronize()
        assert wl.r.status()[0] == 0
        wl.close()
        return
    wl.first_frame()
    K, N, C, T, P = wl.K, wl.N, wl.C, wl.T, wl.P
    M, H, Ht = wl.M, wl.H, wl.Ht
    r, shaded, cam = wl.r, wl.shaded, wl.cam
    image, grads = wl.image, wl.grads
    c_cam, c_prm, bg = wl.c_cam, wl.c_prm, wl.bg

    flush = torch.empty(64 * 1024 * 1024, dtype=torch.int32, device=dev)   # 256 MB > L2

    # ---- CUDA graph of one step
    graph = wl.graph()
    for _ in range(a.warmup):
        flush.zero_()
        graph.replay()
    torch.cuda.synchronize()
    # clocks: the timed steps last milliseconds, shorter than the sampling
    # interval, so the sampler also runs through ~0.4 s of identical steps
    # replayed right before them (the same load; no idle gap)
    clocks = ClockSampler(local)
    clocks.start()
    t_load = time.perf_counter()
    while time.perf_counter() - t_load < 0.4:
        for _ in range(16):
            flush.zero_()
            graph.replay()
        torch.cuda.synchronize()
    if dist:
        dist.barrier()
    torch.cuda.synchronize()
    t_wall0 = time.perf_counter()
    step_ms = time_graph(graph, a.steps, flush)
    t_wall = time.perf_counter() - t_wall0
    clk = clocks.stop()
    if clk:
        clk["window"] = "nvidia-smi every 50 ms over ~0.4 s of identical steps and the timed steps"
    total_ms = max_over_ranks(sum(step_ms), dist, dev)
    if dist:
        dist.barrier()

    # ---- per-stage breakdown (same kernels, eager, events between ABI calls)
    breakdown = wl.breakdown(a.steps, flush)

    # ---- end to end through the API with host buffers (pinned), copies timed.
    # Every step uploads its inputs from pinned host memory and downloads its
    # results.  Pipelined over three streams (the API takes a stream on every
    # call): step i+1's uploads and step i-1's downloads run on the copy
    # engines while step i computes, inputs and outputs double-buffered on the
    # device.  The same steps one at a time are reported as e2e_serial.
    scene = wl.scene
    ins = [("pos", scene.pos), ("radius", scene.radius), ("opacity", scene.opacity),
           ("features", scene.features)]
    ins += [("mlp", wl.mlp_host), ("drgb", wl.drgb_host)] if shaded else [("G", wl.G_host)]
    host_in = {k: torch.from_numpy(np.ascontiguousarray(v)).pin_memory() for k, v in ins}
    host_out = {"image": torch.empty((wl.rgb if shaded else image).shape).pin_memory()}
    for k, v in grads.items():
        host_out[k] = torch.empty(v.shape).pin_memory()
    h2d = sum(v.numel() * 4 for v in host_in.values())
    d2h = sum(v.numel() * 4 for v in host_out.values())
    sets = []
    for _ in range(2):
        st = {"in": {k: torch.empty(v.shape, device=dev) for k, v in host_in.items()},
              "image": torch.empty_like(image),
              "grads": {k: torch.empty_like(v) for k, v in grads.items()}}
        if shaded:
            st["rgb"], st["gF"] = torch.empty_like(wl.rgb), torch.empty_like(wl.gF)
        sets.append(st)

    def compute(st, stream):
        d = st["in"]
        r.render(d["pos"], d["radius"], d["opacity"], d["features"], c_cam, c_prm, bg,
                 image=st["image"], stream=stream)
        if shaded:
            r.shade(st["image"], d["mlp"], st["rgb"], stream=stream)
            r.shade_backward(st["image"], d["mlp"], d["drgb"], st["gF"], st["grads"]["mlp"],
                             stream=stream)
            r.backward(st["gF"], out=st["grads"], stream=stream)
        else:
            r.backward(d["G"], out=st["grads"], stream=stream)

    def download(st):
        host_out["image"].copy_(st["rgb"] if shaded else st["image"], non_blocking=True)
        for k, v in st["grads"].items():
            host_out[k].copy_(v, non_blocking=True)

    s_up, s_cmp, s_dn = (torch.cuda.Stream(device=dev) for _ in range(3))
    ev = {k: [torch.cuda.Event(), torch.cuda.Event()] for k in ("up", "cmp", "dn")}
    # each buffer set's kernels captured once as a CUDA graph (one launch per
    # step; the copies stay explicit on their own streams)
    cgraphs = []
    for st in sets:
        s_cap = torch.cuda.Stream(device=dev)
        s_cap.wait_stream(torch.cuda.current_stream())
        with torch.cuda.stream(s_cap):
            compute(st, s_cap)
        torch.cuda.current_stream().wait_stream(s_cap)
        torch.cuda.synchronize()
        g_ = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g_):
            compute(st, torch.cuda.current_stream())
        cgraphs.append(g_)
    torch.cuda.synchronize()

    def pipelined(n):
        for i in range(n):
            b, st = i & 1, sets[i & 1]
            with torch.cuda.stream(s_up):
                if i >= 2:
                    s_up.wait_event(ev["cmp"][b])   # step i-2 has read these inputs
                for k, v in host_in.items():
                    st["in"][k].copy_(v, non_blocking=True)
                ev["up"][b].record(s_up)
            s_cmp.wait_event(ev["up"][b])
            if i >= 2:
                s_cmp.wait_event(ev["dn"][b])       # step i-2's results are downloaded
            with torch.cuda.stream(s_cmp):
                cgraphs[b].replay()
                ev["cmp"][b].record(s_cmp)
            s_dn.wait_event(ev["cmp"][b])
            with torch.cuda.stream(s_dn):
                download(st)
                ev["dn"][b].record(s_dn)

    def timed_pipelined(n):
        cur = torch.cuda.current_stream()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(cur)
        for s_ in (s_up, s_cmp, s_dn):
            s_.wait_stream(cur)
        pipelined(n)
        for s_ in (s_up, s_cmp, s_dn):
            cur.wait_stream(s_)
        e1.record(cur)
        torch.cuda.synchronize()
        return e0.elapsed_time(e1)

    timed_pipelined(max(2, a.warmup))
    e2e_total = max_over_ranks(timed_pipelined(a.steps), dist, dev)

    def serial_step():
        st = sets[0]
        for k, v in host_in.items():
            st["in"][k].copy_(v, non_blocking=True)
        compute(st, None)
        download(st)

    for _ in range(2):
        serial_step()
    torch.cuda.synchronize()
    serial_ms = []
    for _ in range(a.steps):
        flush.zero_()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        serial_step()
        e1.record()
        torch.cuda.synchronize()
        serial_ms.append(e0.elapsed_time(e1))
    e2e_serial_total = max_over_ranks(sum(serial_ms), dist, dev)
    del cgraphs, sets

    # ---- roofline of the dominant kernel (the forward) and of the whole path
    peaks, peak_src = measured_peaks()
    roofline, path, shade_roof = wl.rooflines(breakdown, total_ms / a.steps, peaks, peak_src, sms)

    value = job_rate(world, K, a.steps, total_ms)   # camera frames (K per step)
    per_cam_loop = None
    if K > 1:
        # the same rig rendered camera by camera through one single-camera
        # context (a graph of K render + backward calls), timed the same way
        r1 = pl.Renderer(max_spheres=N, max_pairs=wl.cap, max_width=cam.width,
                         max_height=cam.height, max_channels=C, max_track=T, device=local)
        singles = [pl.camera(c) for c in wl.cams]
        g1 = {k: (v[0] if k == "cam" else v) for k, v in grads.items()}

        def loop_step():
            for k in range(K):
                r1.render(wl.pos, wl.rad, wl.opa, wl.feat, singles[k], c_prm, bg, image=image[k])
                r1.backward(wl.G[k], out=g1)

        s1 = torch.cuda.Stream(device=dev)
        s1.wait_stream(torch.cuda.current_stream())
        with torch.cuda.stream(s1):
            for _ in range(2):
                loop_step()
        torch.cuda.current_stream().wait_stream(s1)
        torch.cuda.synchronize()
        graph1 = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph1):
            loop_step()
        for _ in range(a.warmup):
            flush.zero_()
            graph1.replay()
        per_cam_loop = sum(time_graph(graph1, a.steps, flush)) / a.steps
        del graph1
        r1.close()
    line = {"metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": a.steps,
            "warmup": a.warmup, "ms_per_step": total_ms / a.steps, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f32", "data": "synthetic",
            "config": {"workload": WORKLOADS[a.scene], "parallelism": f"replicas x{world}",
                       "l2": "flushed between steps (256 MB write, outside the timed events)",
                       "timing": "CUDA events around a CUDA-graph replay of one step"},
            "msphere_pixel_per_s": world * H / (total_ms / a.steps * 1e-3) / 1e6,
            "msphere_pixel_per_s_fwd_bwd": H / ((breakdown["forward"] + breakdown["backward"])
                                                * 1e-3) / 1e6,
            "step_ms_quantiles": {q: float(np.quantile(step_ms, v)) for q, v in
                                  (("p10", 0.1), ("p50", 0.5), ("p90", 0.9))},
            "candidate_tests_per_frame": 256 * M,
            **({"cameras_per_step": K, "camera_by_camera_ms_per_step": per_cam_loop}
               if K > 1 else {}),
            "hits_per_frame": H, "pairs_per_frame": M, "tracked_hits_per_frame": Ht,
            "breakdown_ms": breakdown,
            "path_roofline": path,
            "roofline": roofline,
            **({"shade_roofline": shade_roof} if shaded else {}),
            "e2e": {"value": job_rate(world, K, a.steps, e2e_total), "unit": UNIT,
                    "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                    "timing": "steps pipelined over three streams (uploads of the next and "
                              "downloads of the previous step overlap the current step's "
                              "kernels, replayed from a CUDA graph per buffer set); no L2 "
                              "flush: every step's inputs arrive by copies"},
            "e2e_serial": {"value": job_rate(world, K, a.steps, e2e_serial_total), "unit": UNIT,
                           "timing": "one step at a time: uploads, kernels, downloads in one "
                                     "stream, L2 flushed between steps"},
            "gpu_launches": (KERNELS_PER_STEP + (SHADE_KERNELS if shaded else 0)) * a.steps,
            "clocks": clk, "wall_s_timed": t_wall}
    del graph
    wl.close()
    if a.scene == "headline" and rank == 0 and world == 1 and not a.no_scenes:
        # the other large configurations, timed in the same run the same way
        # (not part of the metric: the headline is)
        line["scenes"] = {name: side_scene(name, dev, local, min(a.steps, 20), 3, flush, peaks,
                                           peak_src, sms)
                          for name in ("neural", "driving")}
    if rank == 0 and world == 1 and not a.no_cpu_baseline:
        shade_args = (wl.mlp_host.astype(np.float64), wl.drgb_host) if shaded else None
        v, rows, dt, cores, reps = oracle_sample(scene, a.cpu_seconds, shade=shade_args)
        what = "fwd, MLP fwd+bwd, bwd" if shaded else "fwd+bwd"
        # the same oracle on one core, on a band sized for a few seconds
        import oracle
        oracle.set_threads(1)
        v1, rows1, dt1, _, _ = oracle_sample(scene, max(2.0, a.cpu_seconds / 4),
                                             rows=max(8, rows // max(1, cores)),
                                             shade=shade_args)
        oracle.set_threads(0)
        line["cpu_baseline_1core"] = {"value": v1, "unit": UNIT, "cores": 1, "kind": "oracle",
                                      "sample": f"rows [0,{rows1}) x 1024 once ({dt1:.1f} s), "
                                                f"scaled by {rows1}/1024"}
        line["cpu_baseline"] = {"value": v, "unit": UNIT, "cores": cores, "kind": "oracle",
                                "sample": f"fp64 oracle {what} on rows [0,{rows}) x 1024 of "
                                          f"the same frame, {reps} time(s) ({dt:.1f} s), "
                                          f"scaled by {rows}/1024"}
    if rank == 0:
        print(json.dumps(line), flush=True)
    if dist:
        dist.destroy_process_group()


def main():
    a = args_parse()
    if a.impl == "reference":
        run_reference(a)
    else:
        run_gb300(a)


if __name__ == "__main__":
    main()
