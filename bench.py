"""Benchmark: 3-D max pooling forward + backward, effective HBM GB/s.

One step = the whole path on one batch: the forward (max + argmax) and the
backward (gradient routing) of the workload, through the C ABI. The timed
workload is the fixed-window k3 s2 fp16 one (32x128x16x112x112 -> 7x55x55):
the largest, and one of the two with a bandwidth target. Other workloads are
reported per kernel under "per_config".

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

Rank 0 prints one JSON line. Under torchrun each rank runs its own shard (an
independent instance of the workload, weak scaling; no collective on the data
path) and the time is the max over ranks.
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

import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

from bwd_maxpool3d_fwd_gb300 import workloads  # noqa: E402

HEADLINE = 3
METRIC = "max-pool3d fwd+bwd effective HBM GB/s and % of GB300 peak, per config"
FALLBACK_HBM_GBS = 6800.0
NOMINAL_HBM_GBS = 8000.0
L2_FLUSH_BYTES = 512 << 20
DTYPE_NAME = {torch.float32: "f32", torch.float16: "f16", torch.bfloat16: "bf16"}


# ---------------------------------------------------------------- bytes

def covered_extent(I, k, s, O, p=0):
    """Input positions along one axis that some window covers (windows start
    at o*s - p and never read padding)."""
    return min(I, (O - 1) * s - p + k) - max(0, -p)


def algorithmic_bytes(w):
    """Minimal bytes: forward = covered input read + y + int64 idx written;
    backward = grad_out + idx read + full grad_in written."""
    es = w.elem_bytes
    P = w.planes
    ovol = w.out[0] * w.out[1] * w.out[2]
    if w.mode == "fixed":
        cov = 1
        for I, k, s, O, p in zip((w.D, w.H, w.W), w.kernel, w.stride, w.out, w.pad):
            cov *= covered_extent(I, k, s, O, p)
    else:
        cov = w.D * w.H * w.W        # adaptive windows cover every input
    vol = w.D * w.H * w.W
    fwd = P * (cov * es + ovol * es + ovol * 8)
    bwd = P * (ovol * es + ovol * 8 + vol * es)
    return fwd, bwd


def hbm_peak():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            v = float(json.load(f)["hbm_gbs"])
        return v, "measured"
    except (OSError, KeyError, ValueError):
        return FALLBACK_HBM_GBS, "fallback"


# ---------------------------------------------------------------- clocks

class ClockSampler:
    """Samples nvidia-smi clocks and throttle reasons while running."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.lines = []
        self.thread = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
            return
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()

    def _read(self):
        for ln in self.proc.stdout:
            self.lines.append(ln.strip())

    def stop(self):
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        if self.thread:
            self.thread.join(timeout=2)
        sm, smax, reasons = [], [], set()
        names = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")
        for ln in self.lines:
            parts = [p.strip() for p in ln.split(",")]
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
            return None
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(smax),
                "reasons": sorted(reasons), "samples": len(sm)}


# ---------------------------------------------------------------- our arm

def channels_last(shape):
    n, c, d, h, w = shape
    return (n, d, h, w, c)


class Runner:
    """Device buffers and the two entry-point calls for one workload, in the
    NCDHW layout or (layout "ndhwc") the channels-last one, where x_cpu and
    g_cpu are given channels-last."""

    def __init__(self, w, x_cpu, g_cpu, dev, algo=None, layout="ncdhw"):
        import bwd_maxpool3d_fwd_gb300 as mp
        self.mp = mp
        self.w = w
        self.dev = dev
        self.layout = layout
        cl = layout == "ndhwc"
        self.x = x_cpu.to(dev)
        self.g = g_cpu.to(dev)
        oshape = channels_last(w.out_shape) if cl else w.out_shape
        self.y = torch.empty(oshape, dtype=w.dtype, device=dev)
        self.idx = torch.empty(oshape, dtype=torch.int64, device=dev)
        self.gin = torch.empty(channels_last(w.in_shape) if cl else w.in_shape, dtype=w.dtype,
                               device=dev)
        self.algo = mp.BWD_AUTO if algo is None else algo
        self.k = w.kernel if w.mode == "fixed" else None
        self.s = w.stride if w.mode == "fixed" else None
        nbytes = mp.maxpool3d_bwd_workspace_bytes(w.in_shape, w.dtype, self.algo)
        self.ws = torch.empty(nbytes // 4, dtype=torch.float32, device=dev) if nbytes else None

    def paths(self):
        mp, w = self.mp, self.w
        if self.layout == "ndhwc":
            return "fwd_ndhwc", mp.maxpool3d_bwd_ndhwc_plan(w.in_shape, w.out, self.k, self.s, w.dtype)
        if any(w.pad):
            return (mp.maxpool3d_fwd_ex_plan(w.in_shape, w.kernel, w.stride, w.pad, (1, 1, 1), False,
                                             w.dtype),
                    mp.maxpool3d_bwd_ex_plan(w.in_shape, w.out, w.kernel, w.stride, w.pad, (1, 1, 1),
                                             False, w.dtype, self.algo))
        if w.mode == "fixed":
            pf = mp.maxpool3d_fwd_plan(w.in_shape, w.kernel, w.stride, w.dtype)
        else:
            pf = mp.adaptive_maxpool3d_fwd_plan(w.in_shape, w.out, w.dtype)
        pb = mp.maxpool3d_bwd_plan(w.in_shape, w.out, self.k, self.s, w.dtype, self.algo)
        return pf, pb

    def launches_per_step(self):
        pf, pb = self.paths()
        nf = 0 if pf == "noop" else 1
        if pb == "noop":
            nb = 0
        elif pb == "bwd_atomic":
            nb = 2 if self.w.dtype == torch.float32 else 3
        else:
            nb = 1
        return nf, nb

    def fwd_values(self):
        """Values-only forward (no index buffer)."""
        if any(self.w.pad):
            self.mp.maxpool3d_fwd_ex(self.x, self.y, None, self.w.kernel, self.w.stride, self.w.pad)
        elif self.w.mode == "fixed":
            self.mp.maxpool3d_fwd(self.x, self.y, None, self.w.kernel, self.w.stride)
        else:
            self.mp.adaptive_maxpool3d_fwd(self.x, self.y, None, self.w.out)

    def fwd(self, x=None, y=None, idx=None):
        x = self.x if x is None else x
        y = self.y if y is None else y
        idx = self.idx if idx is None else idx
        if self.layout == "ndhwc":
            if self.w.mode == "fixed":
                self.mp.maxpool3d_fwd_ndhwc(x, y, idx, self.w.kernel, self.w.stride)
            else:
                self.mp.adaptive_maxpool3d_fwd_ndhwc(x, y, idx, self.w.out)
            return
        if any(self.w.pad):
            self.mp.maxpool3d_fwd_ex(x, y, idx, self.w.kernel, self.w.stride, self.w.pad)
        elif self.w.mode == "fixed":
            self.mp.maxpool3d_fwd(x, y, idx, self.w.kernel, self.w.stride)
        else:
            self.mp.adaptive_maxpool3d_fwd(x, y, idx, self.w.out)

    def bwd(self, g=None, idx=None, gin=None):
        g = self.g if g is None else g
        idx = self.idx if idx is None else idx
        gin = self.gin if gin is None else gin
        if self.layout == "ndhwc":
            self.mp.maxpool3d_bwd_ndhwc(g, idx, gin, self.k, self.s)
            return
        if any(self.w.pad):
            self.mp.maxpool3d_bwd_ex(g, idx, gin, self.k, self.s, self.w.pad, algo=self.algo,
                                     workspace=self.ws)
            return
        self.mp.maxpool3d_bwd(g, idx, gin, self.k, self.s, algo=self.algo, workspace=self.ws)


def l2_flush(buf):
    """Evict the timed kernel's data from L2: write the first half of buf
    (larger than L2), then read the second half (larger than L2), so that the
    flush's own dirty lines are written back before the timed launch and
    not charged to it."""
    n = buf.numel() // 2
    buf[:n].add_(1)
    buf[n:].amax()


def time_per_kernel(r, iters, warmup, flush):
    """Median fwd and bwd device times (ms), each launch preceded by an L2
    flush, CUDA events on the launching stream."""
    stream = torch.cuda.current_stream()
    fb = torch.empty(L2_FLUSH_BYTES // 4, dtype=torch.float32, device=r.dev) if flush else None
    for _ in range(warmup):
        r.fwd()
        r.bwd()
    tf, tb = [], []
    for _ in range(iters):
        for kind, fn, out in (("fwd", r.fwd, tf), ("bwd", r.bwd, tb)):
            if fb is not None:
                l2_flush(fb)
            a = torch.cuda.Event(enable_timing=True)
            b = torch.cuda.Event(enable_timing=True)
            a.record(stream)
            fn()
            b.record(stream)
            b.synchronize()
            out.append(a.elapsed_time(b))
    return statistics.median(tf), statistics.median(tb)


def time_one(fn, dev, iters, flush):
    """Median device time (ms) of fn, each launch preceded by an L2 flush."""
    stream = torch.cuda.current_stream()
    fb = torch.empty(L2_FLUSH_BYTES // 4, dtype=torch.float32, device=dev) if flush else None
    for _ in range(3):
        fn()
    ts = []
    for _ in range(iters):
        if fb is not None:
            l2_flush(fb)
        a = torch.cuda.Event(enable_timing=True)
        b = torch.cuda.Event(enable_timing=True)
        a.record(stream)
        fn()
        b.record(stream)
        b.synchronize()
        ts.append(a.elapsed_time(b))
    return statistics.median(ts)


# Sources each kernel's traffic record depends on (the kernel's file and the
# headers it includes): a record applies only while their hash is the one
# stored with it.
TRAFFIC_SOURCES = {"fwd": ("fwd.cu", "common.cuh", "internal.h"),
                   "bwd": ("bwd_roll.cu", "common.cuh", "internal.h")}


def kernel_hash(kind):
    h = hashlib.sha256()
    for name in TRAFFIC_SOURCES[kind]:
        with open(os.path.join(ROOT, "bwd_maxpool3d_fwd_gb300", "csrc", name), "rb") as f:
            h.update(name.encode() + f.read())
    return h.hexdigest()[:12]


TRAFFIC_WORKLOAD = "fixed_k3s2_f16_32x128x16x112x112"


def recorded_traffic(kernel_kind, workload_name, full):
    """DRAM bytes per launch of the whole workload from the committed ncu
    record (a capture of a subset of planes, scaled by the planes; see the
    record's header), if this run is the whole workload the record is for
    and the kernel's sources are the ones it was taken on; else None."""
    if not full:
        return None
    path = os.path.join(ROOT, "profiles", f"dram_traffic_{workload_name}.txt")
    try:
        with open(path) as f:
            kv = dict(ln.split(":", 1) for ln in f if ":" in ln and not ln.startswith("#"))
    except OSError:
        return None
    kv = {k.strip(): v.strip() for k, v in kv.items()}
    if kv.get(f"{kernel_kind}_sources_sha256_12") != kernel_hash(kernel_kind):
        return None
    v = kv.get(f"{kernel_kind}_dram_bytes_per_launch")
    return int(v) if v else None


# ---------------------------------------------------------------- CPU oracle

def oracle_step(w, x, g):
    """One pass of the oracle over the given planes: forward then backward."""
    import oracle
    if any(w.pad):
        _, idx = oracle.maxpool3d_fwd_ex(x, w.kernel, w.stride, w.pad, (1, 1, 1), False)
    elif w.mode == "fixed":
        _, idx = oracle.maxpool3d_fwd(x, w.kernel, w.stride)
    else:
        _, idx = oracle.adaptive_maxpool3d_fwd(x, w.out)
    oracle.maxpool3d_bwd(g, idx, (w.D, w.H, w.W))


def oracle_sample(w, nplanes):
    planes = list(range(nplanes))
    return workloads.make_x(w, planes=planes), workloads.make_grad_out(w, planes=planes)


def cpu_plane_seconds(w):
    x, g = oracle_sample(w, 4)
    t = time.perf_counter()
    oracle_step(w, x, g)
    return (time.perf_counter() - t) / 4


def cpu_baseline(w, target_s=12.0):
    """The oracle (single-threaded C) on a bounded sample of planes of the
    same workload, sized for about target_s seconds of CPU work."""
    per_plane = cpu_plane_seconds(w)
    n = int(max(1, min(w.planes, target_s / max(per_plane, 1e-6))))
    x, g = oracle_sample(w, n)
    t = time.perf_counter()
    oracle_step(w, x, g)
    dt = time.perf_counter() - t
    fb, bb = algorithmic_bytes(w)
    sample_bytes = (fb + bb) * n / w.planes
    return {"value": round(sample_bytes / dt / 1e9, 4), "unit": "GB/s", "cores": 1,
            "kind": "oracle",
            "sample": f"{n} of {w.planes} planes of {w.name}, forward + backward, "
                      f"{dt:.1f} s on 1 host core (host has {os.cpu_count()} cores)"}


def workload_config(base, layout, world):
    """The `config` object of both arms' JSON lines."""
    return {"workload": base.name, "input": list(base.in_shape),
            "output": list(base.out_shape), "kernel": list(base.kernel),
            "stride": list(base.stride), "padding": list(base.pad), "layout": layout,
            "l2": ("inputs larger than L2 (%d MB input); no flush between steps"
                   % (base.planes * base.D * base.H * base.W * base.elem_bytes // 10**6)),
            "parallelism": f"independent shards x{world}"}


def reference_arm(args):
    """The oracle as the reference implementation, timed on the host cores."""
    w = workloads.by_name_or_index(args.workload)
    if int(os.environ.get("RANK", "0")) != 0:
        return None
    per_plane = cpu_plane_seconds(w)
    budget = 90.0                                  # whole run, seconds
    n = int(max(1, min(w.planes, budget / max(per_plane, 1e-6) / (args.steps + args.warmup))))
    x, g = oracle_sample(w, n)
    for _ in range(args.warmup):
        oracle_step(w, x, g)
    t = time.perf_counter()
    for _ in range(args.steps):
        oracle_step(w, x, g)
    dt = time.perf_counter() - t
    fb, bb = algorithmic_bytes(w)
    step_bytes = (fb + bb) * n / w.planes
    value = step_bytes * args.steps / dt / 1e9
    sample = (f"{n} of {w.planes} planes of {w.name} per step, forward + backward, "
              f"1 host core of {os.cpu_count()}")
    return {"impl": "reference", "metric": METRIC, "value": round(value, 4), "unit": "GB/s",
            "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": round(dt / args.steps * 1e3, 3), "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": DTYPE_NAME[w.dtype],
            "data": "synthetic (seeded)",
            "config": dict(workload_config(w, "ncdhw", 1), planes_per_step=n),
            "cpu_baseline": {"value": round(value, 4), "unit": "GB/s", "cores": 1,
                             "kind": "oracle", "sample": sample},
            "e2e": {"value": round(value, 4), "unit": "GB/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}


# ---------------------------------------------------------------- distributed

def dist_setup():
    """(rank, world, local_rank) from the torchrun environment; a process
    group only when world > 1 (used for a barrier and the max over ranks)."""
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        backend = "nccl" if torch.cuda.is_available() else "gloo"
        if backend == "nccl":
            torch.cuda.set_device(local)
        dist.init_process_group(backend=backend)
    return rank, world, local


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(v: float, world: int, device) -> float:
    if world == 1:
        return v
    import torch.distributed as dist
    t = torch.tensor([v], dtype=torch.float64,
                     device=device if dist.get_backend() == "nccl" else "cpu")
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def shard_seed(w, rank):
    """Each rank's shard is an independent instance of the workload."""
    import dataclasses
    return dataclasses.replace(w, seed=w.seed + 7919 * rank)


def smi_id(dev):
    try:
        p = torch.cuda.get_device_properties(dev)
        return f"{p.pci_domain_id:08X}:{p.pci_bus_id:02X}:{p.pci_device_id:02X}.0"
    except (AttributeError, RuntimeError):
        return str(dev.index or 0)


# ---------------------------------------------------------------- e2e

def e2e(r, x_cpu, g_cpu, steps=8, warmup=2):
    """Same metric through the public API with host buffers: each step copies
    its inputs (x, grad_out) from pinned host memory, runs forward + backward,
    and copies its results (the pooled values y and grad_in) back to pinned
    host memory; the int64 indices stay on the device, where the backward
    consumes them (a caller keeps them there between the two calls). Steps are
    pipelined the way a data loader would run them: two sets of device
    buffers, the copies in, the compute and the copies out on three streams
    ordered by events, so step k + 1's inputs travel while step k computes
    and step k - 1's results come back. The timed region runs from the first
    copy in to the last copy out."""
    w = r.w
    xh, gh = x_cpu.pin_memory(), g_cpu.pin_memory()
    yh = torch.empty(r.y.shape, dtype=w.dtype).pin_memory()
    ginh = torch.empty(r.gin.shape, dtype=w.dtype).pin_memory()
    bufs = [(r.x, r.g, r.y, r.idx, r.gin),
            tuple(torch.empty_like(t) for t in (r.x, r.g, r.y, r.idx, r.gin))]
    s_in, s_cmp, s_out = torch.cuda.Stream(), torch.cuda.Stream(), torch.cuda.Stream()
    ev = lambda: torch.cuda.Event()
    cmp_done = [ev(), ev()]   # compute of the set's last step (it read x, g)
    out_done = [ev(), ev()]   # copies out of the set's last step (they read y, grad_in)
    for e in cmp_done + out_done:
        e.record(torch.cuda.current_stream())

    def step(k):
        x, g, y, idx, gin = bufs[k % 2]
        in_done = ev()
        s_in.wait_event(cmp_done[k % 2])
        with torch.cuda.stream(s_in):
            x.copy_(xh, non_blocking=True)
            g.copy_(gh, non_blocking=True)
            in_done.record(s_in)
        s_cmp.wait_event(in_done)
        s_cmp.wait_event(out_done[k % 2])
        with torch.cuda.stream(s_cmp):
            r.fwd(x, y, idx)
            r.bwd(g, idx, gin)
            cmp_done[k % 2].record(s_cmp)
        s_out.wait_event(cmp_done[k % 2])
        with torch.cuda.stream(s_out):
            yh.copy_(y, non_blocking=True)
            ginh.copy_(gin, non_blocking=True)
            out_done[k % 2].record(s_out)

    for k in range(warmup):
        step(k)
    torch.cuda.synchronize()
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a.record(s_in)
    for k in range(steps):
        step(warmup + k)
    b.record(s_out)
    b.synchronize()
    torch.cuda.synchronize()
    ms = a.elapsed_time(b) / steps
    del bufs
    fb, bb = algorithmic_bytes(w)
    h2d = xh.numel() * xh.element_size() + gh.numel() * gh.element_size()
    d2h = sum(t.numel() * t.element_size() for t in (yh, ginh))
    return {"value": round((fb + bb) / (ms * 1e-3) / 1e9, 2), "unit": "GB/s",
            "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "ms_per_step": round(ms, 3)}


# ---------------------------------------------------------------- main arm

def per_config(dev, peak):
    """Each workload's forward and backward timed alone (median of 20, L2
    flushed before every launch), as GB/s and fraction of the HBM peak."""
    out = {}
    for n, w in enumerate(workloads.WORKLOADS):
        r = Runner(w, workloads.make_x(w), workloads.make_grad_out(w), dev)
        tf, tb = time_per_kernel(r, iters=20, warmup=3, flush=True)
        fb, bb = algorithmic_bytes(w)
        pf, pb = r.paths()
        fg, bg = fb / (tf * 1e-3) / 1e9, bb / (tb * 1e-3) / 1e9
        # values-only forward: the same minus the int64 index writes
        tv = time_one(r.fwd_values, dev, iters=20, flush=True)
        vb = fb - w.planes * w.out[0] * w.out[1] * w.out[2] * 8
        vg = vb / (tv * 1e-3) / 1e9
        # backward without stored indices: timed where the fused 2x2x2 kernel
        # applies (the direct form rescans every covering window per input)
        rec = None
        if w.mode == "fixed" and r.mp.maxpool3d_bwd_recompute_plan(
                w.in_shape, w.out, w.kernel, w.stride, w.dtype) == "bwd_recompute_k2s2":
            tr = time_one(lambda: r.mp.maxpool3d_bwd_recompute(r.x, r.g, r.gin, w.kernel, w.stride),
                          dev, iters=20, flush=True)
            rb = w.planes * (w.D * w.H * w.W * w.elem_bytes * 2 + w.out[0] * w.out[1] * w.out[2] *
                             w.elem_bytes)
            rg = rb / (tr * 1e-3) / 1e9
            rec = {"us": round(tr * 1e3, 2), "bytes": rb, "gbs": round(rg, 1),
                   "frac": round(rg / peak, 4), "path": "bwd_recompute_k2s2"}
        out[w.name] = {
            "fwd_us": round(tf * 1e3, 2), "bwd_us": round(tb * 1e3, 2),
            "fwd_bytes": fb, "bwd_bytes": bb,
            "fwd_gbs": round(fg, 1), "bwd_gbs": round(bg, 1),
            "fwd_frac": round(fg / peak, 4), "bwd_frac": round(bg / peak, 4),
            "fwd_frac_of_nominal_8000": round(fg / NOMINAL_HBM_GBS, 4),
            "bwd_frac_of_nominal_8000": round(bg / NOMINAL_HBM_GBS, 4),
            "fwd_path": pf, "bwd_path": pb,
            "fwd_values_only_us": round(tv * 1e3, 2), "fwd_values_only_bytes": vb,
            "fwd_values_only_gbs": round(vg, 1), "fwd_values_only_frac": round(vg / peak, 4),
            "bwd_recompute": rec}
        del r
        torch.cuda.empty_cache()
    return out


# Padded windows (the padding / dilation / ceil-mode entry points): 3x3x3,
# stride 2, padding 1, fp16, N=8, C=64, 16x56x56 -> 8x28x28. Seeded synthetic
# inputs: x ~ N(0,1) and grad_out ~ N(0,1), drawn in binary32 then rounded.
PADDED = {"name": "padded_k3s2p1_f16_8x64x16x56x56", "shape": (8, 64, 16, 56, 56),
          "k": (3, 3, 3), "s": (2, 2, 2), "p": (1, 1, 1), "dl": (1, 1, 1), "seed": 20261302}
# the same padded window at the size of the k3s2 workload
PADDED_LARGE = {"name": "padded_k3s2p1_f16_32x128x16x112x112", "shape": (32, 128, 16, 112, 112),
                "k": (3, 3, 3), "s": (2, 2, 2), "p": (1, 1, 1), "dl": (1, 1, 1), "seed": 20261303}


def padded_config(dev, peak, c=PADDED):
    """A padded workload's forward and backward timed alone (median of 20,
    L2 flushed before every launch). Inputs are drawn on the device (seeded)."""
    import bwd_maxpool3d_fwd_gb300 as mp
    gen = torch.Generator(device=dev).manual_seed(c["seed"])
    x = torch.randn(c["shape"], generator=gen, device=dev).half()
    out = mp.pool_out_size_ex(c["shape"][2:], c["k"], c["s"], c["p"], c["dl"])
    oshape = c["shape"][:2] + out
    g = torch.randn(oshape, generator=gen, device=dev).half()
    y = torch.empty(oshape, dtype=torch.float16, device=dev)
    idx = torch.empty(oshape, dtype=torch.int64, device=dev)
    gin = torch.empty(c["shape"], dtype=torch.float16, device=dev)
    fwd = lambda: mp.maxpool3d_fwd_ex(x, y, idx, c["k"], c["s"], c["p"], c["dl"])
    bwd = lambda: mp.maxpool3d_bwd_ex(g, idx, gin, c["k"], c["s"], c["p"], c["dl"])
    tf = time_one(fwd, dev, iters=20, flush=True)
    tb = time_one(bwd, dev, iters=20, flush=True)
    nin, nout = x.numel(), y.numel()
    fb, bb = nin * 2 + nout * (2 + 8), nout * (2 + 8) + nin * 2
    fg, bg = fb / (tf * 1e-3) / 1e9, bb / (tb * 1e-3) / 1e9
    return {"fwd_us": round(tf * 1e3, 2), "bwd_us": round(tb * 1e3, 2), "fwd_bytes": fb,
            "bwd_bytes": bb, "fwd_gbs": round(fg, 1), "bwd_gbs": round(bg, 1),
            "fwd_frac": round(fg / peak, 4), "bwd_frac": round(bg / peak, 4),
            "fwd_path": mp.maxpool3d_fwd_ex_plan(c["shape"], c["k"], c["s"], c["p"], c["dl"], False,
                                                 torch.float16),
            "bwd_path": mp.maxpool3d_bwd_ex_plan(c["shape"], out, c["k"], c["s"], c["p"], c["dl"],
                                                 False, torch.float16)}


def ndhwc_configs(dev, peak):
    """The k2s2 and k3s2 workloads in the channels-last layout (the same
    values with the channel axis moved last): forward and backward timed
    alone (median of 20, L2 flushed before every launch)."""
    import bwd_maxpool3d_fwd_gb300 as mp
    out = {}
    for w in workloads.WORKLOADS:
        if w.mode != "fixed":
            continue
        x = workloads.make_x(w).permute(0, 2, 3, 4, 1).contiguous().to(dev)
        g = workloads.make_grad_out(w).permute(0, 2, 3, 4, 1).contiguous().to(dev)
        N, D, H, W, C = x.shape
        oshape = (N,) + tuple(w.out) + (C,)
        y = torch.empty(oshape, dtype=w.dtype, device=dev)
        idx = torch.empty(oshape, dtype=torch.int64, device=dev)
        gin = torch.empty_like(x)
        tf = time_one(lambda: mp.maxpool3d_fwd_ndhwc(x, y, idx, w.kernel, w.stride), dev, 20, True)
        tb = time_one(lambda: mp.maxpool3d_bwd_ndhwc(g, idx, gin, w.kernel, w.stride), dev, 20, True)
        fb, bb = algorithmic_bytes(w)
        fg, bg = fb / (tf * 1e-3) / 1e9, bb / (tb * 1e-3) / 1e9
        out[w.name + "_ndhwc"] = {
            "fwd_us": round(tf * 1e3, 2), "bwd_us": round(tb * 1e3, 2), "fwd_bytes": fb,
            "bwd_bytes": bb, "fwd_gbs": round(fg, 1), "bwd_gbs": round(bg, 1),
            "fwd_frac": round(fg / peak, 4), "bwd_frac": round(bg / peak, 4),
            "fwd_path": "fwd_ndhwc",
            "bwd_path": mp.maxpool3d_bwd_ndhwc_plan((N, C, D, H, W), w.out, w.kernel, w.stride, w.dtype)}
        del x, g, y, idx, gin
        torch.cuda.empty_cache()
    return out


def our_arm(args):
    rank, world, local = dist_setup()
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    import bwd_maxpool3d_fwd_gb300 as mp
    mp.lib()                                     # fail loudly if the library is missing
    base = workloads.by_name_or_index(args.workload)
    cl = args.layout == "ndhwc"
    if args.planes:
        import dataclasses
        if cl:   # whole samples: the channel axis stays whole
            base = dataclasses.replace(base, N=max(1, min(base.N, args.planes // base.C)))
        else:
            base = dataclasses.replace(base, N=1, C=min(args.planes, base.planes))
    w = shard_seed(base, rank)
    x_cpu, g_cpu = workloads.make_x(w), workloads.make_grad_out(w)
    if cl:
        x_cpu = x_cpu.permute(0, 2, 3, 4, 1).contiguous()
        g_cpu = g_cpu.permute(0, 2, 3, 4, 1).contiguous()
    r = Runner(w, x_cpu, g_cpu, dev, layout=args.layout)
    peak, peak_kind = hbm_peak()
    fb, bb = algorithmic_bytes(w)
    nf, nb = r.launches_per_step()
    stream = torch.cuda.current_stream()

    for _ in range(args.warmup):
        r.fwd()
        r.bwd()
    torch.cuda.synchronize()
    sampler = ClockSampler(smi_id(dev)) if rank == 0 else None
    if sampler:
        sampler.start()
        time.sleep(1.0)
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True),
           torch.cuda.Event(enable_timing=True)) for _ in range(args.steps)]
    barrier(world)
    torch.cuda.synchronize()
    t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    t0.record(stream)
    for e0, e1, e2 in ev:
        e0.record(stream)
        r.fwd()
        e1.record(stream)
        r.bwd()
        e2.record(stream)
    t1.record(stream)
    torch.cuda.synchronize()
    barrier(world)
    clocks = sampler.stop() if sampler else None
    total_ms = max_over_ranks(t0.elapsed_time(t1), world, dev)
    fwd_ms = statistics.mean(a.elapsed_time(b) for a, b, _ in ev)
    bwd_ms = statistics.mean(b.elapsed_time(c) for _, b, c in ev)

    step_bytes = fb + bb
    value = step_bytes * args.steps * world / (total_ms * 1e-3) / 1e9
    kind, kbytes, kms = ("bwd", bb, bwd_ms) if bwd_ms >= fwd_ms else ("fwd", fb, fwd_ms)
    pf, pb = r.paths()
    achieved = kbytes / (kms * 1e-3) / 1e9
    roofline = {"bound": "hbm", "achieved": round(achieved, 1), "peak": peak, "unit": "GB/s",
                "frac": round(achieved / peak, 4),
                "traffic": recorded_traffic(kind, w.name, not args.planes and not cl),
                "kernel": pb if kind == "bwd" else pf, "peak_source": peak_kind,
                "bytes_per_launch": kbytes,
                "fwd": {"path": pf, "us": round(fwd_ms * 1e3, 2), "bytes": fb,
                        "gbs": round(fb / (fwd_ms * 1e-3) / 1e9, 1),
                        "frac": round(fb / (fwd_ms * 1e-3) / 1e9 / peak, 4)},
                "bwd": {"path": pb, "us": round(bwd_ms * 1e3, 2), "bytes": bb,
                        "gbs": round(bb / (bwd_ms * 1e-3) / 1e9, 1),
                        "frac": round(bb / (bwd_ms * 1e-3) / 1e9 / peak, 4)}}
    e2e_res = None if args.no_e2e else e2e(r, x_cpu, g_cpu)
    del r
    torch.cuda.empty_cache()
    cfg = per_config(dev, peak) if (rank == 0 and not args.no_per_config) else None
    if cfg is not None:
        cfg[PADDED["name"]] = padded_config(dev, peak)
        cfg[PADDED_LARGE["name"]] = padded_config(dev, peak, PADDED_LARGE)
        torch.cuda.empty_cache()
        cfg.update(ndhwc_configs(dev, peak))
    cpu = cpu_baseline(base) if (rank == 0 and world == 1 and not args.no_cpu_baseline) else None
    if rank != 0:
        return None
    return {
        "metric": METRIC, "value": round(value, 2), "unit": "GB/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(total_ms / args.steps, 4), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": DTYPE_NAME[w.dtype],
        "data": "synthetic (seeded generators; shapes and value recipes of the workload)",
        "config": workload_config(base, args.layout, world),
        "roofline": roofline, "cpu_baseline": cpu, "e2e": e2e_res,
        "gpu_launches": (nf + nb) * args.steps, "clocks": clocks,
        "per_config": cfg,
    }


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=1500)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", choices=("ours", "reference"), default="ours")
    ap.add_argument("--workload", default=str(HEADLINE),
                    help="index of one of the five workloads, or a workload name (e.g. "
                         "fixed_k3s2p1_f16_32x128x16x112x112, the padded form of workload 3)")
    ap.add_argument("--no-per-config", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true",
                    help="skip the end-to-end leg (its second set of device buffers); for profiling")
    ap.add_argument("--planes", type=int, default=0,
                    help="run only the first N planes of the workload (same per-plane shape; "
                         "for profiling small cases; whole samples with --layout ndhwc)")
    ap.add_argument("--layout", choices=("ncdhw", "ndhwc"), default="ncdhw",
                    help="tensor layout of the timed step (ndhwc: the channels-last entry points)")
    args = ap.parse_args(argv)
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    res = reference_arm(args) if args.impl == "reference" else our_arm(args)
    if res is not None:
        print(json.dumps(res), flush=True)


if __name__ == "__main__":
    main()
