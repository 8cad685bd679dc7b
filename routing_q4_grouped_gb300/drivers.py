"""Command-line drivers of single library calls on the seeded synthetic inputs,
for profilers (ncu) and quick timings.

    python -m routing_q4_grouped_gb300.drivers layer  T [calls]   # moe_layer, full-width layer
    python -m routing_q4_grouped_gb300.drivers router T [calls]   # moe_router_topk

The full-width layer has d = 2048, 256 experts, top-8, f = f_s = 512 and the
value recipe of the t512 workload; T tokens of its seeded x and logits. Each
call goes through the C-ABI on the current stream; the driver prints the mean
time of the calls after the first (CUDA events) and the device error word.
"""
from __future__ import annotations

import dataclasses
import sys

import numpy as np
import torch

from . import moeq4, synth


def _layer(T: int, calls: int) -> None:
    cfg = dataclasses.replace(synth.CONFIGS["t512"], T=T)
    W = moeq4.DeviceWeights.from_host(synth.gen_weights(cfg, 0))
    x = torch.from_numpy(synth.gen_x(cfg, T).view(np.int16)).cuda().view(torch.bfloat16)
    lg = torch.from_numpy(synth.gen_logits(cfg, 0, T)).cuda()
    lay = moeq4.Layer(W, T, cfg.k, None)
    _timed(lambda: lay(x, lg), calls, lay.route)


def _router(T: int, calls: int) -> None:
    cfg = dataclasses.replace(synth.CONFIGS["t4096"], T=T)
    x = torch.from_numpy(synth.gen_x(cfg, T).view(np.int16)).cuda().view(torch.bfloat16)
    wr = torch.from_numpy(synth.gen_router(cfg).view(np.int16)).cuda().view(torch.bfloat16)
    out = moeq4.RouteBuffers.alloc(T, cfg.E, cfg.k, 128)
    lg = torch.empty((T, cfg.E), dtype=torch.float32, device="cuda")
    _timed(lambda: moeq4.moe_router_topk(x, wr, out, lg), calls, out)


def _timed(fn, calls: int, route) -> None:
    fn()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    for _ in range(calls - 1):
        fn()
    e1.record()
    torch.cuda.synchronize()
    us = e0.elapsed_time(e1) / max(1, calls - 1) * 1e3
    print(f"mean {us:.1f} us per call over {calls - 1} calls; device error word "
          f"{moeq4.moe_get_device_error(route)}")


def main(argv) -> None:
    what, T = argv[1], int(argv[2])
    calls = int(argv[3]) if len(argv) > 3 else 4
    {"layer": _layer, "router": _router}[what](T, calls)


if __name__ == "__main__":
    main(sys.argv)
