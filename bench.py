"""Benchmark of the W4A16 NVFP4 MoE layer on GB300 (one JSON line on rank 0).

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference] [--workload NAME]
                    [--workloads grouped,prefill,skewed]

A step is one pass of the whole layer (route -> permute -> gate_up+SwiGLU ->
down -> combine) over one batch of seeded synthetic input of the decode-shaped
workload (T=32 tokens, H=2048, I=768, 128 experts, top-8, NVFP4 weights).

ours:      inputs resident in HBM; each timed step is moe_layer_forward_profiled
           (same kernels as moe_layer_forward) bracketed by CUDA events on the
           launching stream, the L2 flushed between steps (a 2x-L2 buffer written, then a
           second 2x-L2 buffer read so that the flush's own write-backs finish before the step)
           outside the events.  `e2e` runs a caller-owned host plan (moe_host_plan_run):
           pinned host x / logits in, host out back, copies inside the timed region.
           The other workloads of the metric (grouped: the Atlas article's 800 tokens x
           256 experts; prefill; skewed), and all four through the block-scaled FP4
           (W4A4) layer (keys ending in _w4a4), are timed the same way after the
           headline one and reported under "workloads".
reference: the fp64 CPU oracle (single thread) on a bounded token sample of the
           same workload; rank 0 only.
N > 1 ranks run independent replicas (the path needs no exchange between GPUs);
value = tokens of all ranks / max-over-ranks time.
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

import numpy as np
import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

from moe_layer_bit_gb300 import workloads as wk  # noqa: E402

METRIC = "MoE-layer tokens/s at 1 GB300; HBM GB/s (decode) / tensor TFLOP/s (prefill) vs peak"
UNIT = "tokens/s"
DEFAULT_WORKLOAD = "decode"


def _peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            p = json.load(f)
        return float(p["hbm_gbs"]), float(p["bf16_tflops"]), float(p["bf16_tflops_sustained"]), "measured"
    except Exception:
        return 6800.0, 1900.0, 1700.0, "fallback"


# ------------------------------------------------------------------- clocks
class ClockSampler:
    """SM clock and clock-event (throttle) reasons sampled while the timed region runs.

    Read-only NVML queries (nvmlDeviceGetClockInfo / GetCurrentClocksEventReasons)
    every ~1 ms from a thread, so even a timed region of a few milliseconds gets
    samples; falls back to `nvidia-smi -lms 100` when NVML cannot be loaded."""
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")
    # nvmlClocksEventReason* bits
    REASON_BITS = {0x4: "sw_power_cap", 0x8: "hw_slowdown", 0x20: "sw_thermal_slowdown",
                   0x40: "hw_thermal_slowdown", 0x80: "hw_power_brake_slowdown"}

    def __init__(self, device):
        self.device = device
        self.proc = None
        self.lines = []
        self.thread = None
        self.nvml = None
        self.handle = None
        self.samples = []
        self.stop_flag = threading.Event()

    def _open_nvml(self):
        import ctypes
        try:
            lib = ctypes.CDLL("libnvidia-ml.so.1")
        except OSError:
            return False
        if lib.nvmlInit_v2() != 0:
            return False
        h = ctypes.c_void_p()
        ok = False
        try:
            u = str(torch.cuda.get_device_properties(self.device).uuid)
            u = u if u.startswith("GPU-") else "GPU-" + u
            ok = lib.nvmlDeviceGetHandleByUUID(u.encode(), ctypes.byref(h)) == 0
        except Exception:
            ok = False
        if not ok:
            vis = os.environ.get("CUDA_VISIBLE_DEVICES", "")
            idx = self.device.index or 0
            if vis and vis.split(",")[idx].strip().isdigit():
                idx = int(vis.split(",")[idx])
            ok = lib.nvmlDeviceGetHandleByIndex_v2(ctypes.c_uint(idx), ctypes.byref(h)) == 0
        if not ok:
            return False
        self.reasons_fn = getattr(lib, "nvmlDeviceGetCurrentClocksEventReasons", None) or \
            getattr(lib, "nvmlDeviceGetCurrentClocksThrottleReasons")
        self.nvml, self.handle = lib, h
        return True

    def _poll(self):
        import ctypes
        clk, mx, rs = ctypes.c_uint(), ctypes.c_uint(), ctypes.c_ulonglong()
        while not self.stop_flag.is_set():
            a = self.nvml.nvmlDeviceGetClockInfo(self.handle, 1, ctypes.byref(clk))        # NVML_CLOCK_SM
            b = self.nvml.nvmlDeviceGetMaxClockInfo(self.handle, 1, ctypes.byref(mx))
            c = self.reasons_fn(self.handle, ctypes.byref(rs))
            if a == 0 and b == 0 and c == 0:
                self.samples.append((clk.value, mx.value, rs.value))
            time.sleep(0.001)

    def start(self):
        if self._open_nvml():
            self.thread = threading.Thread(target=self._poll, daemon=True)
            self.thread.start()
            return
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.device.index or 0), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
            return
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def stop(self):
        sm, smax, reasons = [], [], set()
        if self.nvml is not None:
            self.stop_flag.set()
            self.thread.join(timeout=2)
            for c, m, r in self.samples:
                sm.append(float(c))
                smax.append(float(m))
                for bit, nm in self.REASON_BITS.items():
                    if r & bit:
                        reasons.add(nm)
            src = "nvml"
        elif self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
            self.thread.join(timeout=2)
            names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
            for ln in self.lines:
                parts = [p.strip() for p in ln.split(",")]
                if len(parts) < 9:
                    continue
                try:
                    sm.append(float(parts[1]))
                    smax.append(float(parts[2]))
                except ValueError:
                    continue
                for nm, v in zip(names, parts[5:9]):
                    if v.lower() == "active":
                        reasons.add(nm)
            src = "nvidia-smi"
        else:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no clock source"], "samples": 0}
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(smax) if smax else None,
                "reasons": sorted(reasons), "samples": len(sm), "source": src}


# ------------------------------------------------------------ distributed
def _dist_init(args):
    world = int(os.environ.get("WORLD_SIZE", "1"))
    if world > 1:
        import torch.distributed as dist
        backend = "nccl" if torch.cuda.is_available() and args.impl == "ours" else "gloo"
        dist.init_process_group(backend=backend)
        return dist, int(os.environ.get("RANK", "0")), world, int(os.environ.get("LOCAL_RANK", "0"))
    return None, 0, 1, 0


def _max_over_ranks(dist, v: float, device) -> float:
    if dist is None:
        return v
    t = torch.tensor([v], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def _job_throughput(dist, world: int, tokens_per_rank: int, seconds: float, device) -> float:
    """Whole-job tokens/s of N replicas: the tokens all ranks processed over the
    slowest rank's time."""
    return world * tokens_per_rank / _max_over_ranks(dist, seconds, device)


def _barrier(dist, device=None):
    if dist is not None:
        if device is not None and device.type == "cuda":
            dist.barrier(device_ids=[device.index])
        else:
            dist.barrier()


# --------------------------------------------------------------- CPU oracle
def oracle_sample(d, wl, n_tokens: int, seed: int = 0):
    """Time the fp64 oracle on a seeded token sample; returns (seconds, n_tokens)."""
    from oracle import oracle as orc
    rng = np.random.default_rng(seed)
    rows = np.sort(rng.choice(wl.T, size=min(n_tokens, wl.T), replace=False)).astype(np.int32)
    xb = d["x"].view(torch.int16).numpy().view(np.uint16)
    gu = tuple(a.numpy() for a in d["gu"])
    dn = tuple(a.numpy() for a in d["dn"])
    t0 = time.perf_counter()
    ids, w = orc.route(d["logits"].numpy(), wl.k)
    orc.layer_rows(xb, ids, w, gu, dn, rows)
    return time.perf_counter() - t0, len(rows)


def _oracle_tokens_for(wl, seconds: float) -> int:
    per_token_macs = wl.k * 3 * wl.H * wl.I
    est = 5.0e8  # fp64 decode + multiply-add per second on one core (measured order of magnitude)
    return int(max(1, min(wl.T, round(seconds * est / per_token_macs))))


def oracle_baseline(d, wl, budget_s: float):
    """Repeat seeded oracle samples until about budget_s of CPU time; returns (seconds, tokens, reps, n)."""
    n = _oracle_tokens_for(wl, min(budget_s, 5.0))
    total, toks, reps = 0.0, 0, 0
    while total < budget_s or reps < 1:
        dt, nt = oracle_sample(d, wl, n, seed=reps)
        total += dt
        toks += nt
        reps += 1
    return total, toks, reps, n


NOMINAL_HBM_GBS = 7900.0  # GB300 nominal HBM3e bandwidth, for context beside the measured copy peak
EXTRA_WORKLOADS = ("grouped", "prefill", "skewed", "decode:w4a4", "grouped:w4a4", "prefill:w4a4", "skewed:w4a4")


def bench_config(wl, world: int) -> dict:
    """The `config` object of both arms' JSON lines (same keys, same values)."""
    return {"workload": wl.name, "T": wl.T, "H": wl.H, "I": wl.I, "E": wl.E, "k": wl.k,
            "parallelism": f"replicas x{world}" if world > 1 else "single",
            "l2": "flushed between steps, outside the timed events: a 2x-L2 buffer written, then another "
                  "2x-L2 buffer read (the flush's dirty lines reach HBM before the step)"}


def run_reference(args, wl, dist, rank, world):
    if rank != 0:
        return
    d = wk.generate(wl)
    n = _oracle_tokens_for(wl, args.ref_step_seconds)
    for _ in range(min(args.warmup, 1)):
        oracle_sample(d, wl, max(1, n // 4), seed=99)
    total, toks = 0.0, 0
    for s in range(args.steps):
        dt, nt = oracle_sample(d, wl, n, seed=s)
        total += dt
        toks += nt
    value = toks / total
    sample = f"{n} of {wl.T} tokens per step (seeded), full routing of all {wl.T} tokens, fp64, 1 thread"
    line = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": args.gpus, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": 1e3 * total / args.steps, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic (seeded)",
        "config": bench_config(wl, world if world > 1 else args.gpus),
        "impl": "reference",
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": 1, "kind": "oracle", "sample": sample},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


# ------------------------------------------------------------------ ours
W4A16_SOURCES = ("gemm_w4a16.cu", "gemm_common.cuh", "device_common.cuh")
W4A4_SOURCES = ("gemm_w4a4.cu", "gemm_common.cuh", "device_common.cuh")


def _kernel_hash(files=W4A16_SOURCES) -> str:
    h = hashlib.sha256()
    for f in files:
        with open(os.path.join(ROOT, "moe_layer_bit_gb300", "csrc", f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:16]


def _traffic_from_profile(wl, prefix="gemm_", files=W4A16_SOURCES):
    """Per-launch DRAM bytes of the dominant GEMM launch from the committed ncu summary, or None
    if the summary is missing or was taken on a different kernel source."""
    p = os.path.join(ROOT, "profiles", f"{prefix}{wl.name}.txt")
    if not os.path.exists(p):
        return None
    kv = {}
    with open(p) as f:
        for line in f:
            if ":" in line and not line.startswith("#"):
                k, v = line.split(":", 1)
                kv[k.strip()] = v.strip()
    if kv.get("kernel_source_sha256_16") != _kernel_hash(files):
        return None
    try:
        return float(kv["dram_bytes_per_launch"])
    except (KeyError, ValueError):
        return None


class DeviceBench:
    """One workload on one GPU: the layer built from seeded inputs, an L2 flush
    between steps, and CUDA events on the launching stream."""

    def __init__(self, wl, dev, rank):
        from moe_layer_bit_gb300 import _lib
        from moe_layer_bit_gb300.layer import MoELayer
        self.lib = _lib
        self.wl, self.dev = wl, dev
        self.d = wk.generate(wl, seed=wl.seed + rank)
        self.layer = MoELayer(self.d["gu"], self.d["dn"], wl.H, wl.I, wl.E, wl.k, wl.T, dev)
        self.x = self.d["x"].to(dev)
        self.logits = self.d["logits"].to(dev)
        self.out = torch.empty(wl.T, wl.H, dtype=torch.bfloat16, device=dev)
        self.ids = torch.empty(wl.T, wl.k, dtype=torch.int32, device=dev)
        self.tw = torch.empty(wl.T, wl.k, dtype=torch.float32, device=dev)
        self.dims = self.layer.dims(wl.T)
        l2 = getattr(torch.cuda.get_device_properties(dev), "L2_cache_size", 126 * 2 ** 20)
        self.flush = torch.empty(2 * l2 // 4 + 1024, dtype=torch.float32, device=dev)
        self.clean = torch.ones(2 * l2 // 4 + 1024, dtype=torch.float32, device=dev)
        self.stream = torch.cuda.current_stream(dev)

    def flush_l2(self, v):
        # Write a 2x-L2 buffer (evicts everything the layer touched), then read
        # another 2x-L2 buffer, so the written lines are back in HBM before the
        # next step instead of being written back during it.
        self.flush.fill_(v)
        return self.clean.sum()

    def step(self, evs):
        self.lib.moe_layer_forward_profiled(self.x, self.logits, self.layer.w_gate_up.abi, self.layer.w_down.abi,
                                            self.dims, self.out, self.ids, self.tw, self.layer.ws,
                                            self.layer.ws_bytes, evs, self.stream)

    def check_status(self, when):
        st = self.layer.device_status()
        if st != self.lib.MOE_OK:
            raise RuntimeError(f"{self.wl.name}: device status {when}: {self.lib.status_string(st)}")

    def _events(self, steps):
        evs = [[torch.cuda.Event(enable_timing=True) for _ in range(6)] for _ in range(steps)]
        # torch only reports elapsed time between events it has recorded itself; record
        # each once here (the library records them again inside every timed step)
        for e in evs:
            for ev in e:
                ev.record(self.stream)
        return evs

    def _timed_region(self, dist, evs, stage_marks):
        """K steps; the L2 flush sits between steps, outside the events.  With
        stage_marks False only the step's first and last events are recorded, so
        nothing separates the layer's kernels (their programmatic launch overlap
        is kept); with True all six are, for the per-stage times."""
        _barrier(dist, self.dev)
        torch.cuda.synchronize(self.dev)
        t0 = time.perf_counter()
        for s in range(len(evs)):
            self.flush_l2(float(s))
            e = evs[s] if stage_marks else [evs[s][0], None, None, None, None, evs[s][5]]
            self.step(e)
        torch.cuda.synchronize(self.dev)
        _barrier(dist, self.dev)
        return time.perf_counter() - t0

    def measure(self, steps, warmup, dist, world):
        wl = self.wl
        warm_evs = [torch.cuda.Event(enable_timing=True) for _ in range(6)]
        for _ in range(warmup):
            self.flush_l2(1.0)
            self.step(warm_evs)
        torch.cuda.synchronize(self.dev)
        self.check_status("after warm-up")
        evs = self._events(steps)
        stage_evs = self._events(steps)
        torch.cuda.synchronize(self.dev)
        clocks = ClockSampler(self.dev)
        clocks.start()
        t_wall = self._timed_region(dist, evs, False)           # the measured steps
        t_wall_stages = self._timed_region(dist, stage_evs, True)  # the same steps again, per-stage events
        clk = clocks.stop()
        self.check_status("after timing")
        step_ms = [e[0].elapsed_time(e[5]) for e in evs]
        stage_ms = np.array([[e[i].elapsed_time(e[i + 1]) for i in range(5)] for e in stage_evs])
        total_s = sum(step_ms) / 1e3
        value = _job_throughput(dist, world, wl.T * steps, total_s, self.dev)
        counts = np.bincount(self.ids.cpu().numpy().reshape(-1), minlength=wl.E)
        touched = int(np.count_nonzero(counts))
        mean_step_ms = total_s * 1e3 / steps
        roofline = self.roofline(stage_ms, touched)
        layer_bytes = wk.algorithmic_bytes(wl.T, wl.H, wl.I, wl.E, wl.k, counts)
        layer_flops = wk.algorithmic_flops(wl.T, wl.H, wl.I, wl.k)
        hbm_peak, tf_peak, _, _ = _peaks()
        return {
            "value": value, "unit": UNIT, "ms_per_step": mean_step_ms, "steps": steps, "warmup": warmup,
            "touched_experts": touched, "layer_bytes": layer_bytes, "layer_flops": layer_flops,
            "roofline": roofline,
            "layer_roofline": {"achieved_gbs": layer_bytes / (mean_step_ms * 1e-3) / 1e9,
                               "frac_hbm": layer_bytes / (mean_step_ms * 1e-3) / 1e9 / hbm_peak,
                               "achieved_tflops": layer_flops / (mean_step_ms * 1e-3) / 1e12,
                               "frac_tensor": layer_flops / (mean_step_ms * 1e-3) / 1e12 / tf_peak},
            "stages_ms": {nm: float(stage_ms[:, i].mean()) for i, nm in
                          enumerate(["route_group", "gather", "gate_up_swiglu", "down", "combine"])},
            "wall_s_timed_loop": t_wall, "wall_s_stage_loop": t_wall_stages,
            "gpu_launches": self.lib.moe_layer_kernel_launches(self.dims) * steps,
            "clocks": clk,
        }

    def roofline(self, stage_ms, touched):
        """Roofline of the dominant kernel: gate_up + SwiGLU, or both projections
        when the layer runs them as one launch (then stage 2 spans that launch and
        stage 3 is empty).  Algorithmic bytes / flops per launch over the launch's
        mean event-timed duration; the bound is the roof it is closer to."""
        wl = self.wl
        n = wl.T * wl.k
        fused = self.lib.moe_layer_projections_fused(self.dims)
        gu_bytes = touched * (2 * wl.I * wl.H * 9 // 16 + 4) + n * wl.H * 2 + n * wl.I * 2
        if fused:
            gu_bytes += touched * (wl.H * wl.I * 9 // 16 + 4) + n * wl.I * 2 + n * wl.H * 4
        gu_ms = float(stage_ms[:, 2].mean())
        hbm_peak, tf_peak, tf_sus, peak_kind = _peaks()
        achieved = gu_bytes / (gu_ms * 1e-3) / 1e9
        gu_flops = 2 * n * (3 if fused else 2) * wl.I * wl.H
        achieved_tf = gu_flops / (gu_ms * 1e-3) / 1e12
        if achieved_tf / tf_peak > achieved / hbm_peak:
            r = {"bound": "tensor", "achieved": achieved_tf, "peak": tf_peak, "unit": "TFLOP/s",
                 "frac": achieved_tf / tf_peak, "peak_kind": f"{peak_kind} burst cuBLAS bf16 GEMM",
                 "frac_sustained_peak": achieved_tf / tf_sus, "algorithmic_flops_per_launch": gu_flops}
        else:
            r = {"bound": "hbm", "achieved": achieved, "peak": hbm_peak, "unit": "GB/s",
                 "frac": achieved / hbm_peak, "peak_kind": f"{peak_kind} burst copy bandwidth",
                 "frac_nominal_7900": achieved / NOMINAL_HBM_GBS, "algorithmic_bytes_per_launch": gu_bytes}
        r.update({"kernel": "w4a16_gemm_kernel (gate_up + SwiGLU" + (", then down, one launch)" if fused else ")"),
                  "traffic": _traffic_from_profile(wl),
                  "launch_ms": gu_ms,
                  "other_roof_frac": (achieved / hbm_peak) if r["bound"] == "tensor" else (achieved_tf / tf_peak)})
        if not fused:
            dn_ms = float(stage_ms[:, 3].mean())
            dn_bytes = touched * (wl.H * wl.I * 9 // 16 + 4) + n * wl.I * 2 + n * wl.H * 4
            dn_flops = 2 * n * wl.I * wl.H
            r["down"] = {"launch_ms": dn_ms, "achieved_gbs": dn_bytes / (dn_ms * 1e-3) / 1e9,
                         "frac_hbm": dn_bytes / (dn_ms * 1e-3) / 1e9 / hbm_peak,
                         "achieved_tflops": dn_flops / (dn_ms * 1e-3) / 1e12,
                         "frac_tensor": dn_flops / (dn_ms * 1e-3) / 1e12 / tf_peak}
        return r

    def stream_probe(self, nbytes_alg, steps):
        """What one kernel of the GEMM's shape reads in the same time budget when it
        does nothing else: the streaming probe over the same byte count, same flush."""
        nbytes = (nbytes_alg // 18432) * 18432
        probe_buf = torch.empty(nbytes, dtype=torch.uint8, device=self.dev)
        pev = [[torch.cuda.Event(enable_timing=True) for _ in range(2)] for _ in range(steps)]
        for _ in range(3):
            self.flush_l2(0.0)
            self.lib.moe_debug_stream_read(probe_buf, nbytes, self.layer.ws, self.stream)
        for st in range(steps):
            self.flush_l2(float(st))
            pev[st][0].record(self.stream)
            self.lib.moe_debug_stream_read(probe_buf, nbytes, self.layer.ws, self.stream)
            pev[st][1].record(self.stream)
        torch.cuda.synchronize(self.dev)
        self.check_status("after the stream probe")
        probe_ms = float(np.mean([e[0].elapsed_time(e[1]) for e in pev]))
        return {"what": "one CTA per SM, 8 x 18432-byte bulk copies in flight, nothing else; same byte count "
                        "and L2 flush", "bytes": nbytes, "ms": probe_ms, "gbs": nbytes / (probe_ms * 1e-3) / 1e9}

    def e2e(self, steps, warmup, dist, world):
        """End to end through the public host-buffer API: a caller-owned host plan
        on page-locked x / logits / out and a stream of its own; each step copies x
        host->device, the routing kernel reads the logits and the combine writes the
        output through their mapped addresses, and the call synchronises."""
        wl = self.wl
        xh = self.d["x"].pin_memory()
        lh = self.d["logits"].pin_memory()
        oh = torch.empty(wl.T, wl.H, dtype=torch.bfloat16).pin_memory()
        e2e_stream = torch.cuda.Stream(self.dev)
        times = []
        with self.layer.host_plan(xh, lh, oh, e2e_stream) as plan:
            for _ in range(max(3, warmup)):
                plan.run()
            for s in range(steps):
                self.flush_l2(float(s))
                torch.cuda.synchronize(self.dev)
                t0 = time.perf_counter()
                plan.run()  # synchronises before returning
                times.append(time.perf_counter() - t0)
        self.check_status("after the host-plan steps")
        value = _job_throughput(dist, world, wl.T * steps, sum(times), self.dev)
        return {"value": value, "unit": UNIT, "h2d_bytes_per_step": wl.T * wl.H * 2 + wl.T * wl.E * 4,
                "d2h_bytes_per_step": wl.T * wl.H * 2, "api": "moe_host_plan_run (page-locked host buffers)"}

    def close(self):
        del self.layer, self.x, self.logits, self.out, self.flush, self.clean
        torch.cuda.synchronize(self.dev)
        torch.cuda.empty_cache()


FP4_OVER_BF16 = 13.5 / 2.25  # nominal dense FP4 / BF16 tensor rate of GB300


class W4A4Bench(DeviceBench):
    """The same measurement for the block-scaled FP4 layer (NVFP4 activations,
    tcgen05 kind::mxf4nvf4); its roofline is taken against the FP4 tensor peak
    (the measured bf16 peak times the nominal FP4 / BF16 ratio)."""

    def __init__(self, wl, dev, rank):
        from moe_layer_bit_gb300 import _lib
        from moe_layer_bit_gb300.layer import W4A4Layer
        self.lib = _lib
        self.wl, self.dev = wl, dev
        self.d = wk.generate(wl, seed=wl.seed + rank)
        self.layer = W4A4Layer(self.d["gu"], self.d["dn"], wl.H, wl.I, wl.E, wl.k, wl.T, dev)
        self.x = self.d["x"].to(dev)
        self.logits = self.d["logits"].to(dev)
        self.out = torch.empty(wl.T, wl.H, dtype=torch.bfloat16, device=dev)
        self.ids = torch.empty(wl.T, wl.k, dtype=torch.int32, device=dev)
        self.tw = torch.empty(wl.T, wl.k, dtype=torch.float32, device=dev)
        self.dims = _lib.dims(wl.T, wl.H, wl.I, wl.E, wl.k)
        l2 = getattr(torch.cuda.get_device_properties(dev), "L2_cache_size", 126 * 2 ** 20)
        self.flush = torch.empty(2 * l2 // 4 + 1024, dtype=torch.float32, device=dev)
        self.clean = torch.ones(2 * l2 // 4 + 1024, dtype=torch.float32, device=dev)
        self.stream = torch.cuda.current_stream(dev)

    def step(self, evs):
        self.lib.moe_layer_forward_w4a4_profiled(self.x, self.logits, self.layer._abi[0], self.layer._abi[1],
                                                 self.dims, self.out, self.ids, self.tw, self.layer.ws,
                                                 self.layer.ws_bytes, evs, self.stream)

    def measure(self, steps, warmup, dist, world):
        m = super().measure(steps, warmup, dist, world)
        m["gpu_launches"] = self.lib.moe_w4a4_kernel_launches(self.dims) * steps
        lr = m["layer_roofline"]
        lr["frac_tensor_fp4"] = lr.pop("frac_tensor") / FP4_OVER_BF16
        m["stages_ms"] = dict(zip(["route_group", "quantize_gather", "gate_up_swiglu", "down", "combine"],
                                  m["stages_ms"].values()))
        return m

    def roofline(self, stage_ms, touched):
        wl = self.wl
        n = wl.T * wl.k
        _, tf_peak, tf_sus, peak_kind = _peaks()
        fp4_peak, fp4_sus = tf_peak * FP4_OVER_BF16, tf_sus * FP4_OVER_BF16
        hbm_peak = _peaks()[0]
        gu_ms, dn_ms = float(stage_ms[:, 2].mean()), float(stage_ms[:, 3].mean())
        gu_flops, dn_flops = 4 * n * wl.H * wl.I, 2 * n * wl.H * wl.I
        # NVFP4 weights of the touched experts, x's NVFP4 rows read, h's written (9/16 B per element)
        gu_bytes = touched * (2 * wl.I * wl.H * 9 // 16 + 4) + n * wl.H * 9 // 16 + n * wl.I * 9 // 16
        dn_bytes = touched * (wl.H * wl.I * 9 // 16 + 4) + n * wl.I * 9 // 16 + n * wl.H * 4
        a = gu_flops / (gu_ms * 1e-3) / 1e12
        ab = gu_bytes / (gu_ms * 1e-3) / 1e9
        if a / fp4_peak > ab / hbm_peak:
            r = {"bound": "tensor", "achieved": a, "peak": fp4_peak, "unit": "TFLOP/s", "frac": a / fp4_peak,
                 "frac_sustained_peak": a / fp4_sus,
                 "peak_kind": f"{peak_kind} burst cuBLAS bf16 GEMM x {FP4_OVER_BF16:g} (nominal dense FP4 / BF16)",
                 "algorithmic_flops_per_launch": gu_flops}
        else:
            r = {"bound": "hbm", "achieved": ab, "peak": hbm_peak, "unit": "GB/s", "frac": ab / hbm_peak,
                 "peak_kind": f"{peak_kind} burst copy bandwidth", "frac_nominal_7900": ab / NOMINAL_HBM_GBS,
                 "algorithmic_bytes_per_launch": gu_bytes}
        r.update({"launch_ms": gu_ms, "kernel": "w4a4_gemm_kernel (gate_up + SwiGLU + NVFP4 quantization of h)",
                  "traffic": _traffic_from_profile(wl, "gemm_w4a4_", W4A4_SOURCES),
                  "other_roof_frac": (ab / hbm_peak) if r["bound"] == "tensor" else (a / fp4_peak),
                  "down": {"launch_ms": dn_ms, "achieved_gbs": dn_bytes / (dn_ms * 1e-3) / 1e9,
                           "frac_hbm": dn_bytes / (dn_ms * 1e-3) / 1e9 / hbm_peak,
                           "achieved_tflops": dn_flops / (dn_ms * 1e-3) / 1e12,
                           "frac_tensor_fp4": dn_flops / (dn_ms * 1e-3) / 1e12 / fp4_peak}})
        return r


def run_ours(args, wl, dist, rank, world, local_rank):
    from moe_layer_bit_gb300 import _lib, build

    if not torch.cuda.is_available():
        raise RuntimeError("bench.py --impl ours needs a CUDA device")
    dev = torch.device("cuda", local_rank)
    torch.cuda.set_device(dev)
    if rank == 0:
        build.build()
    _barrier(dist)
    _lib.load()

    b = DeviceBench(wl, dev, rank)
    m = b.measure(args.steps, args.warmup, dist, world)
    roofline = m["roofline"]
    if roofline["bound"] == "hbm":
        probe = b.stream_probe(roofline["algorithmic_bytes_per_launch"], args.steps)
        probe["kernel_vs_probe"] = roofline["achieved"] / probe["gbs"]
        roofline["stream_probe"] = probe
    e2e = b.e2e(args.steps, args.warmup, dist, world)

    # ---- CPU oracle baseline on a bounded sample (rank 0, N = 1 only)
    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        dt, nt, reps, n_tok = oracle_baseline(b.d, wl, args.cpu_seconds)
        cpu = {"value": nt / dt, "unit": UNIT, "cores": 1, "kind": "oracle",
               "sample": f"{reps} x {n_tok} of {wl.T} tokens (seeded) after routing all {wl.T}; fp64, "
                         f"single thread, {dt:.1f} s"}
    b.close()

    # ---- the other workloads of the metric, same method, same run (context lines, not the headline)
    extra = {}
    names = [n for n in (EXTRA_WORKLOADS if args.workloads is None else args.workloads.split(",")) if n]
    for name in names:
        w4a4 = name.endswith(":w4a4")
        xwl = wk.by_name(name.split(":")[0])
        if xwl.name == wl.name and not w4a4:
            continue
        xb = (W4A4Bench if w4a4 else DeviceBench)(xwl, dev, rank)
        xm = xb.measure(args.steps, args.warmup, dist, world)
        xm["config"] = dict(bench_config(xwl, world), path="w4a4" if w4a4 else "w4a16")
        extra[xwl.name + ("_w4a4" if w4a4 else "")] = xm
        xb.close()

    if rank != 0:
        return
    line = {
        "metric": METRIC, "value": m["value"], "unit": UNIT, "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": m["ms_per_step"], "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16 x nvfp4 (fp32 accumulate)", "data": "synthetic (seeded, random-init)",
        "config": bench_config(wl, world),
        "workload_detail": {"touched_experts": m["touched_experts"], "layer_bytes": m["layer_bytes"],
                            "layer_flops": m["layer_flops"]},
        "roofline": roofline,
        "layer_roofline": m["layer_roofline"],
        "stages_ms": m["stages_ms"],
        "wall_s_timed_loop": m["wall_s_timed_loop"],
        "wall_s_stage_loop": m["wall_s_stage_loop"],
        "e2e": e2e,
        "cpu_baseline": cpu,
        # the library's own kernels per step (routing + grouping, row gather unless the
        # GEMM gathers, gate_up, down, combine) times the timed steps
        "gpu_launches": m["gpu_launches"],
        "clocks": m["clocks"],
        "workloads": extra,
    }
    print(json.dumps(line), flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=50)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default=DEFAULT_WORKLOAD)
    ap.add_argument("--cpu-seconds", type=float, default=12.0, help="target length of the CPU oracle sample")
    ap.add_argument("--ref-step-seconds", type=float, default=1.5)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--workloads", default=None,
                    help="comma-separated extra workloads timed after the headline one (default: "
                         + ",".join(EXTRA_WORKLOADS) + "; '' for none)")
    args = ap.parse_args()
    if args.warmup < 3 and args.impl == "ours":
        ap.error("--warmup must be >= 3")
    wl = wk.by_name(args.workload)
    dist, rank, world, local_rank = _dist_init(args)
    try:
        if args.impl == "reference":
            run_reference(args, wl, dist, rank, world)
        else:
            run_ours(args, wl, dist, rank, world, local_rank)
    finally:
        if dist is not None:
            dist.destroy_process_group()


if __name__ == "__main__":
    main()
