"""Choose the grouped GEMM's token-tile width and tile schedule by measurement.

    python -m moe_layer_bit_gb300.tune [--workloads decode,grouped,prefill,skewed] [--steps K] [--warmup W]

For each workload (the seeded synthetic inputs of workloads.py) and each
combination of token-tile width (16, 32, 64, 128 rows) and tile schedule
(static persistent, claim persistent, the Atlas article's 3-D grid
(ceil(N/BN), max token tiles, experts)), runs the whole layer through
moe_debug_layer_forward_config and times it with CUDA events on the launching
stream, the L2 flushed between steps (outside the events).  Prints one JSON
line per combination (mean ms per layer call, tokens/s, the GEMM stages' times,
whether the output is bit-identical to the library's default choice) and a
final line naming the fastest combination per workload.  The library's
default choice (plan_layer in csrc/gemm_w4a16.cu) is set from these numbers.
"""
from __future__ import annotations

import argparse
import json

import numpy as np
import torch

from . import _lib, build
from . import workloads as wk
from .layer import MoELayer

SCHEDULES = {0: "static", 1: "claim", 2: "grid3d"}
TILES = (16, 32, 64, 128)


def _time(layer, x, logits, out, dims, bn, sched, steps, warmup, flush, clean, stream):
    """Mean ms per layer call with only the first and last events recorded (the
    kernels' programmatic launch overlap is kept), then the per-stage means
    from a second pass with all six events."""
    def run(evs):
        _lib.moe_debug_layer_forward_config(x, logits, layer.w_gate_up.abi, layer.w_down.abi, dims, out, None, None,
                                            layer.ws, layer.ws_bytes, bn, sched, evs, stream)

    def events():
        evs = [[torch.cuda.Event(enable_timing=True) for _ in range(6)] for _ in range(steps)]
        for e in evs:
            for ev in e:
                ev.record(stream)
        return evs

    warm = [torch.cuda.Event(enable_timing=True) for _ in range(6)]
    for _ in range(warmup):
        flush.fill_(1.0)
        clean.sum()
        run(warm)
    torch.cuda.synchronize()
    whole, staged = events(), events()
    for s in range(steps):
        flush.fill_(float(s))
        clean.sum()
        run([whole[s][0], None, None, None, None, whole[s][5]])
    for s in range(steps):
        flush.fill_(float(s))
        clean.sum()
        run(staged[s])
    torch.cuda.synchronize()
    st = layer.device_status()
    if st != _lib.MOE_OK:
        raise RuntimeError(f"device status {_lib.status_string(st)} for bn={bn} sched={sched}")
    ms = float(np.mean([e[0].elapsed_time(e[5]) for e in whole]))
    stage = np.array([[e[i].elapsed_time(e[i + 1]) for i in range(5)] for e in staged])
    return ms, stage.mean(axis=0)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--workloads", default="decode,grouped,prefill,skewed")
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--tiles", default="16,32,64,128")
    ap.add_argument("--schedules", default="0,1,2")
    args = ap.parse_args()
    build.build()
    _lib.load()
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    l2 = getattr(torch.cuda.get_device_properties(dev), "L2_cache_size", 126 * 2 ** 20)
    flush = torch.empty(2 * l2 // 4 + 1024, dtype=torch.float32, device=dev)
    clean = torch.ones(2 * l2 // 4 + 1024, dtype=torch.float32, device=dev)
    stream = torch.cuda.current_stream(dev)
    best = {}
    for name in args.workloads.split(","):
        wl = wk.by_name(name)
        d = wk.generate(wl)
        layer = MoELayer(d["gu"], d["dn"], wl.H, wl.I, wl.E, wl.k, wl.T, dev)
        x, logits = d["x"].to(dev), d["logits"].to(dev)
        dims = layer.dims(wl.T)
        ref = torch.empty(wl.T, wl.H, dtype=torch.bfloat16, device=dev)
        layer.forward(x, logits, out=ref)
        out = torch.empty_like(ref)
        for bn in [int(t) for t in args.tiles.split(",")]:
            for sched in [int(v) for v in args.schedules.split(",")]:
                try:
                    ms, stage = _time(layer, x, logits, out, dims, bn, sched, args.steps, args.warmup, flush, clean,
                                      stream)
                except _lib.MoeError as e:
                    print(json.dumps({"workload": wl.name, "token_tile": bn, "schedule": SCHEDULES[sched],
                                      "error": str(e)}), flush=True)
                    continue
                same = bool(torch.equal(out.view(torch.int16), ref.view(torch.int16)))
                row = {"workload": wl.name, "token_tile": bn, "schedule": SCHEDULES[sched], "ms": ms,
                       "tokens_per_s": wl.T / (ms * 1e-3),
                       "stages_ms": dict(zip(["route_group", "gather", "gemm0", "gemm1", "combine"],
                                             [float(v) for v in stage])),
                       "bit_identical_to_default": same}
                print(json.dumps(row), flush=True)
                if wl.name not in best or ms < best[wl.name]["ms"]:
                    best[wl.name] = {"token_tile": bn, "schedule": SCHEDULES[sched], "ms": ms}
        del layer
        torch.cuda.empty_cache()
    print(json.dumps({"fastest": best}), flush=True)


if __name__ == "__main__":
    main()
