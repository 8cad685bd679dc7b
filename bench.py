#!/usr/bin/env python3
"""Benchmark of the prefill MoE expert layer (routing + 4-bit grouped GEMM).

    python bench.py [--gpus N --steps K --warmup W] [--impl ours|reference]
                    [--workload t4096] [--block-m 128]

One step = one full MoE layer call (routing, gate/up pass, down pass with the
combine and the bf16 output) over one batch of T tokens of synthetic input already resident in
HBM. Steps cycle through independent layer sets (weights, x, logits) whose
weights alone exceed the 129 MB L2. Prints ONE JSON line on rank 0.

Under torchrun (N > 1) every rank runs its own replica on its own GPU (the
layer is independent per token batch: weak scaling, no data-path collective);
the time is the max over ranks.

--workload chunked runs the chunked multi-layer prefill instead: one step is
T = 32768 tokens in 4096-token chunks through 40 layers with their own weights
(routing, both GEMM passes and the next-input step per chunk and layer).

The default run also measures the other single-layer workloads (t512, skew,
tiny) in the same process and reports them under "workloads", and times the
CPU oracle on one whole layer over the host cores ("cpu_baseline").

--impl reference times the CPU oracle (plain numpy, float64) on the same
workload on the host cores: every step is one whole layer (one chunk-layer
for the chunked run), its expert groups spread over one worker process per
core.
"""
import os

# The CPU baseline is the oracle as it stands, one BLAS thread per process
# (fixed before numpy loads, inherited by the worker processes), so that
# "cores" is the number of processes it really used.
for _v in ("OMP_NUM_THREADS", "OPENBLAS_NUM_THREADS", "MKL_NUM_THREADS"):
    os.environ.setdefault(_v, "1")

import argparse
import hashlib
import json
import re
import statistics
import subprocess
import sys
import tempfile
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "MoE-layer prefill tokens/s at T=4096; grouped-GEMM % of GB300 BF16 TC peak"
UNIT = "tokens/s"
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}
# stage events 0..5 bracket: routing (one or two launches; events 1 and 2 coincide),
# gate/up GEMM, down GEMM with the combine and the bf16 output (events 4 and 5
# coincide)
STAGES = ["route", None, "gemm_gate_up_swiglu", "gemm_down_combine", None]


def launches_per_layer(T, decode=False):
    """Kernel launches of one moe_layer call: routing takes one launch when one
    block covers the batch (T <= 8) and two otherwise; the FFN two (the grouped
    GEMM's passes) or three on the small-batch path (gate/up, down, bf16 output)."""
    return (1 if T <= 8 else 2) + (3 if decode else 2)

KERNEL_SOURCES = ["gemm.cu", "dequant.cuh", "ptx.cuh"]


def parse_args():
    p = argparse.ArgumentParser()
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=20)
    p.add_argument("--warmup", type=int, default=5)
    p.add_argument("--impl", choices=["ours", "reference"], default="ours")
    p.add_argument("--workload", default="t4096")
    p.add_argument("--block-m", default="auto",
                   help="tile rows of the block map; auto = 64 for short expert groups, else 128")
    p.add_argument("--sets", type=int, default=2, help="independent layer sets cycled per step")
    p.add_argument("--no-cpu-baseline", action="store_true")
    p.add_argument("--prefetch-mb", type=int, default=32,
                   help="chunked run: MB of the next layer's weights prefetched into L2 during "
                        "each layer's tail (0 = off)")
    p.add_argument("--no-workloads", action="store_true",
                   help="time only --workload (not the other single-layer workloads)")
    return p.parse_args()


def peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            d = json.load(f)
        return d, "measured"
    return FALLBACK_PEAKS, "fallback"


def kernel_source_hash():
    h = hashlib.sha256()
    for n in KERNEL_SOURCES:
        with open(os.path.join(ROOT, "routing_q4_grouped_gb300", "csrc", n), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def profiled_traffic(workload):
    """DRAM bytes per launch of the gate/up kernel from the committed ncu summary
    of this workload (the gate/up kernel's own summary, else the summary of all
    the layer's kernels), if it was taken on the current kernel sources (else None)."""
    for name in (f"gemm_gate_up_{workload}.md", f"layer_kernels_{workload}.md"):
        path = os.path.join(ROOT, "profiles", name)
        if os.path.exists(path):
            break
    else:
        return None
    txt = open(path).read()
    m = re.search(r"traffic_bytes_per_launch:\s*([0-9]+)", txt)
    hm = re.search(r"kernel_source_sha:\s*([0-9a-f]+)", txt)
    if not m or not hm or hm.group(1) != kernel_source_hash():
        return None
    return int(m.group(1))


class ClockSampler:
    """nvidia-smi clock / throttle sampling during the timed region."""

    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index):
        self.idx = gpu_index
        self.proc = None
        self.path = None

    def start(self):
        try:
            fd, self.path = tempfile.mkstemp(suffix=".csv")
            os.close(fd)
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.idx}", f"--query-gpu={self.Q}", "--format=csv,noheader,nounits",
                 "-lms", "100"], stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        rows = []
        for line in open(self.path):
            parts = [x.strip() for x in line.split(",")]
            if len(parts) >= 9:
                rows.append(parts)
        os.unlink(self.path)
        if not rows:
            return None

        def num(x):
            try:
                return float(x)
            except ValueError:
                return None

        sm = [num(r[1]) for r in rows if num(r[1]) is not None]
        smax = [num(r[2]) for r in rows if num(r[2]) is not None]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in rows for i in range(4) if r[5 + i].lower() == "active"})
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(smax) if smax else None, "reasons": reasons,
                "samples": len(rows)}


def dist_setup():
    import torch

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist

        torch.cuda.set_device(local)
        dist.init_process_group("nccl")
    else:
        torch.cuda.set_device(0)
    return world, rank, local


def barrier(world):
    if world > 1:
        import torch.distributed as dist

        dist.barrier()


def max_over_ranks(world, v):
    """Largest v over the ranks (NCCL: a device tensor; gloo: a host tensor)."""
    if world == 1:
        return v
    import torch
    import torch.distributed as dist

    dev = "cuda" if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([v], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def layer_ids(rank, sets):
    """Synthetic layer seeds of a rank's layer sets: every rank runs its own replica
    on its own inputs (rank r: layers r*sets .. r*sets + sets - 1)."""
    return [rank * sets + i for i in range(sets)]


# ----------------------------------------------------------------- CPU oracle
#
# The oracle as it stands (plain numpy, float64, one BLAS thread per process),
# timed on the host cores: whole layers, their expert groups spread over one
# spawned worker process per core (oracle.pool); routing runs in the parent,
# inside the timed region.


def host_cores():
    try:
        n = len(os.sched_getaffinity(0))
    except AttributeError:  # pragma: no cover
        n = os.cpu_count() or 1
    return max(1, min(n, 64))


def oracle_single_core_sample(cfg, W, x, logits, block_m, n_groups=4):
    """Single-process oracle on a bounded sample: routing of all T tokens plus
    the FFN of n_groups expert groups of about the mean size, scaled by rows to
    one full layer. Returns (seconds for the full layer, note)."""
    import oracle as O

    T = x.shape[0]
    t0 = time.perf_counter()
    r = O.route(logits, cfg.k, block_m)
    t_route = time.perf_counter() - t0
    near = np.argsort(np.abs(r.counts - r.counts.mean()), kind="stable")[:n_groups]
    groups = [int(g) for g in near]
    rows = int(sum(r.counts[g] for g in groups))
    t0 = time.perf_counter()
    O.expert_ffn(x, W, r, experts=groups, shared=False)
    t_ffn = time.perf_counter() - t0
    total_rows = T * cfg.k + (T if cfg.f_s else 0)
    full = t_route + t_ffn * total_rows / rows
    note = (f"routing of all {T} tokens + FFN of {len(groups)} expert groups ({rows} of "
            f"{total_rows} rows incl. shared), scaled by rows to one full layer")
    return full, note


def oracle_baseline(cfg, block_m, steps=1, warmup=0, procs=None):
    """The oracle on whole layers of the workload (one chunk-layer for the
    chunked run) over `procs` host processes. Returns a dict with the mean
    seconds per layer, the per-layer times and the process count."""
    from routing_q4_grouped_gb300 import synth

    procs = procs or host_cores()
    T = cfg.tokens_per_call
    W = synth.gen_weights(cfg, 0)
    x = synth.gen_x(cfg, T)
    logits = synth.gen_logits(cfg, 0, T)
    from oracle.pool import OraclePool

    pool = OraclePool(procs)
    try:
        pool.load(W, x)
        for _ in range(warmup):
            pool.layer(logits, cfg.k, block_m)
        times = []
        for _ in range(steps):
            t0 = time.perf_counter()
            pool.layer(logits, cfg.k, block_m)
            times.append(time.perf_counter() - t0)
    finally:
        pool.close()
    single, single_note = oracle_single_core_sample(cfg, W, x, logits, block_m)
    return {"sec": statistics.mean(times), "times": times, "procs": procs,
            "single_core_sec": single, "single_core_note": single_note}


def run_reference(args):
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return
    from routing_q4_grouped_gb300 import synth

    cfg = synth.CONFIGS[args.workload]
    T = cfg.tokens_per_call
    b = oracle_baseline(cfg, args.block_m, steps=args.steps, warmup=args.warmup)
    sec = b["sec"]
    if cfg.layers > 1:
        # a step is one chunk-layer of the chunked run (4096 tokens through one
        # layer); the run's tokens/s follows from its layers x chunks such steps
        n_chunks = cfg.T // T
        value = cfg.T / (sec * cfg.layers * n_chunks)
        sample = (f"per step: one whole chunk-layer ({T} tokens through one layer, routing + "
                  f"every expert group + shared expert) over {b['procs']} processes; the run's "
                  f"tokens/s = {cfg.T} tokens / ({cfg.layers} layers x {n_chunks} chunks x "
                  f"the measured step time)")
    else:
        value = T / sec
        sample = (f"per step: one whole layer ({T} tokens, routing + every expert group + "
                  f"shared expert) over {b['procs']} processes")
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": sec * 1e3,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic (seeded generator, same recipe as the GPU arm)",
        "config": workload_config(cfg, args, world),
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": b["procs"], "kind": "oracle",
                         "sample": sample,
                         "single_core": {"value": T / b["single_core_sec"] if cfg.layers == 1 else
                                         cfg.T / (b["single_core_sec"] * cfg.layers * (cfg.T // T)),
                                         "unit": UNIT, "cores": 1,
                                         "sample": b["single_core_note"]}},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def workload_config(cfg, args, world):
    c = {"workload": args.workload, "T": cfg.T, "d": cfg.d, "E": cfg.E, "k": cfg.k, "f": cfg.f,
         "f_s": cfg.f_s, "block_m": args.block_m, "parallelism": f"replicas x{world}"}
    if cfg.layers > 1:
        c.update(chunk=cfg.chunk, layers=cfg.layers)
    else:
        c.update(layer_sets=args.sets)
    return c


# ---------------------------------------------------------------------- GPU arm


def layer_bytes(cfg, T, touched):
    """Algorithmic bytes of one layer call: the 4-bit weights of the touched
    experts and of the shared expert (0.5 B per weight + 4 B per 64 weights),
    x and y in bf16 and the fp32 logits."""
    d, f, fs, E = cfg.d, cfg.f, cfg.f_s, cfg.E
    per_expert = 3 * d * f // 2 + 3 * d * f // 64 * 4
    shared = 3 * d * fs // 2 + 3 * d * fs // 64 * 4
    return touched * per_expert + shared + 2 * T * d * 2 + T * E * 4


def measure_workload(name, args, world, rank, local, steps, warmup, sets_n, clocks_on=True,
                     block_m=None):
    """Times the layer on workload `name` (steps cycling through sets_n
    independent layer sets) and returns the measured figures."""
    import torch

    from routing_q4_grouped_gb300 import moeq4, synth

    cfg = synth.CONFIGS[name]
    T, d, E, k, f, fs = cfg.tokens_per_call, cfg.d, cfg.E, cfg.k, cfg.f, cfg.f_s
    bm = block_m or moeq4.default_block_m(T, E, k)
    stream = torch.cuda.current_stream()

    sets = []
    for layer in layer_ids(rank, sets_n):
        W = moeq4.DeviceWeights.from_host(synth.gen_weights(cfg, layer))
        x_h = synth.gen_x(cfg, T, layer)
        l_h = synth.gen_logits(cfg, layer, T)
        x = torch.from_numpy(x_h.view(np.int16)).cuda().view(torch.bfloat16)
        lg = torch.from_numpy(l_h).cuda()
        sets.append((W, x, lg, x_h, l_h))
    route = moeq4.RouteBuffers.alloc(T, E, k, bm)
    ws = moeq4.alloc_workspace(moeq4.moe_layer_workspace_size(T, E, k, d, f, fs, bm))
    y = torch.empty((T, d), dtype=torch.bfloat16, device="cuda")
    weight_bytes = sets[0][0].nbytes

    def step(i):
        W, x, lg = sets[i % len(sets)][:3]
        moeq4.moe_layer(x, lg, W, route, y, ws, stream)

    for i in range(warmup):
        step(i)
    torch.cuda.synchronize()
    if moeq4.moe_get_device_error(route) != 0:
        raise RuntimeError("device error word set during warm-up")

    # ---- timed region: K steps, inputs resident in HBM
    clocks = ClockSampler(local) if clocks_on else None
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    barrier(world)
    torch.cuda.synchronize()
    if clocks:
        clocks.start()
        time.sleep(0.3)  # let the sampler start
    ev0.record(stream)
    for i in range(steps):
        step(i)
    ev1.record(stream)
    torch.cuda.synchronize()
    clk = clocks.stop() if clocks else None
    barrier(world)
    ms_total = max_over_ranks(world, ev0.elapsed_time(ev1))
    ms_step = ms_total / steps
    value = T * world * steps / (ms_total * 1e-3)

    # ---- per-kernel times over the same K steps, stage events on the launching stream
    stage_ms = {s: [] for s in STAGES if s}
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(6)] for _ in range(steps)]
    for row in evs:             # torch creates the CUDA event on first record
        for e in row:
            e.record(stream)
    torch.cuda.synchronize()
    for i in range(steps):
        moeq4.moe_debug_set_stage_events(evs[i])
        step(i)
    moeq4.moe_debug_set_stage_events([])
    torch.cuda.synchronize()
    for i in range(steps):
        for j, s in enumerate(STAGES):
            if s:
                stage_ms[s].append(evs[i][j].elapsed_time(evs[i][j + 1]))
    kern = {s: statistics.mean(v) for s, v in stage_ms.items()}

    # ---- end to end through the public call: every step copies its x and logits
    # from pinned host memory, runs the layer and copies y back to pinned host
    # memory. Copies run on their own streams (host->device, device->host) into
    # double-buffered device slots, so step i's copies overlap the layers of
    # steps i-1 and i+1; events order every slot's reuse.
    pins = [(torch.from_numpy(s[3].view(np.int16)).pin_memory(),
             torch.from_numpy(s[4]).pin_memory()) for s in sets]
    x_dev = [torch.empty_like(sets[0][1]) for _ in range(2)]
    l_dev = [torch.empty_like(sets[0][2]) for _ in range(2)]
    y_dev = [torch.empty((T, d), dtype=torch.bfloat16, device="cuda") for _ in range(2)]
    y_host = [torch.empty((T, d), dtype=torch.int16).pin_memory() for _ in range(2)]
    h2d_s, d2h_s = torch.cuda.Stream(), torch.cuda.Stream()
    in_ready = [torch.cuda.Event() for _ in range(2)]
    in_free = [torch.cuda.Event() for _ in range(2)]
    out_ready = [torch.cuda.Event() for _ in range(2)]
    out_free = [torch.cuda.Event() for _ in range(2)]
    for b in range(2):       # all slots start free
        in_free[b].record(stream)
        out_free[b].record(d2h_s)

    def e2e_step(i):
        b = i % 2
        xh, lh = pins[i % len(pins)]
        with torch.cuda.stream(h2d_s):
            h2d_s.wait_event(in_free[b])
            x_dev[b].view(torch.int16).copy_(xh, non_blocking=True)
            l_dev[b].copy_(lh, non_blocking=True)
            in_ready[b].record(h2d_s)
        stream.wait_event(in_ready[b])
        stream.wait_event(out_free[b])
        moeq4.moe_layer(x_dev[b], l_dev[b], sets[i % len(sets)][0], route, y_dev[b], ws, stream)
        in_free[b].record(stream)
        out_ready[b].record(stream)
        with torch.cuda.stream(d2h_s):
            d2h_s.wait_event(out_ready[b])
            y_host[b].copy_(y_dev[b].view(torch.int16), non_blocking=True)
            out_free[b].record(d2h_s)

    for i in range(2):
        e2e_step(i)
    torch.cuda.synchronize()
    barrier(world)
    ev0.record(stream)
    h2d_s.wait_event(ev0)
    for i in range(steps):
        e2e_step(i)
    done = torch.cuda.Event()
    done.record(d2h_s)
    stream.wait_event(done)
    ev1.record(stream)
    torch.cuda.synchronize()
    e2e_ms = max_over_ranks(world, ev0.elapsed_time(ev1))
    e2e_value = T * world * steps / (e2e_ms * 1e-3)
    h2d = T * d * 2 + T * E * 4
    d2h = T * d * 2

    if moeq4.moe_get_device_error(route) != 0:
        raise RuntimeError("device error word set during the timed region")

    # ---- rooflines: the dominant kernel (the gate/up pass), the grouped GEMM and the layer
    pk, pk_src = peaks()
    flops_gu = 4 * d * f * T * k + 4 * d * fs * T
    flops_dn = 2 * d * f * T * k + 2 * d * fs * T
    counts = route.counts.cpu().numpy()
    touched = int((counts > 0).sum())
    per_expert_gu = 2 * f * d // 2 + 2 * f * (d // 64) * 4
    sh_gu = 2 * fs * d // 2 + 2 * fs * (d // 64) * 4
    bytes_gu = touched * per_expert_gu + sh_gu + T * d * 2 + T * k * f * 2 + T * fs * 2
    peak_tf = pk["bf16_tflops"]
    peak_gb = pk["hbm_gbs"]
    t_gu = kern["gemm_gate_up_swiglu"] * 1e-3
    t_dn = kern["gemm_down_combine"] * 1e-3
    if flops_gu / (peak_tf * 1e12) >= bytes_gu / (peak_gb * 1e9):
        roof = {"bound": "tensor", "achieved": flops_gu / t_gu / 1e12, "peak": peak_tf,
                "unit": "TFLOP/s"}
    else:
        roof = {"bound": "hbm", "achieved": bytes_gu / t_gu / 1e9, "peak": peak_gb, "unit": "GB/s"}
    roof["frac"] = roof["achieved"] / roof["peak"]
    roof["traffic"] = profiled_traffic(name)
    roof["kernel"] = "q4_grouped_gemm_kernel<0> (gate/up + SwiGLU)"
    roof["peak_source"] = f"{pk_src} (bf16 burst / hbm copy)"
    gg_tflops = (flops_gu + flops_dn) / (t_gu + t_dn) / 1e12
    # the whole layer against the slower of its FLOPs at the bf16 peak and its
    # algorithmic bytes at the copy bandwidth
    lb = layer_bytes(cfg, T, touched)
    lf = flops_gu + flops_dn
    t_roof = max(lf / (peak_tf * 1e12), lb / (peak_gb * 1e9))
    layer_roof = {"bound": "tensor" if lf / (peak_tf * 1e12) >= lb / (peak_gb * 1e9) else "hbm",
                  "flops": lf, "bytes": lb, "roofline_us": t_roof * 1e6,
                  "achieved_gbs": lb / (ms_step * 1e-3) / 1e9,
                  "achieved_tflops": lf / (ms_step * 1e-3) / 1e12,
                  "frac": t_roof / (ms_step * 1e-3)}
    return {
        "cfg": cfg, "T": T, "block_m": bm, "value": value, "ms_per_step": ms_step,
        "kernels_ms": kern, "roofline": roof, "layer_roofline": layer_roof,
        "grouped_gemm": {"tflops": gg_tflops, "frac_bf16_peak": gg_tflops / peak_tf,
                         "ms": (t_gu + t_dn) * 1e3},
        "touched_experts": touched,
        "e2e": {"value": e2e_value, "unit": UNIT, "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": d2h},
        "clocks": clk, "weight_bytes": weight_bytes, "launches": launches_per_layer(T) * steps,
    }


def measure_router(name, steps, warmup):
    """The fused router (projection + top-k) alone and the whole layer from
    hidden states (router, routing from its choice, expert FFN) on workload
    `name`, with seeded router weights ~ N(0, 1/d)."""
    import torch

    from routing_q4_grouped_gb300 import moeq4, synth

    cfg = synth.CONFIGS[name]
    T, d, E, k, f, fs = cfg.tokens_per_call, cfg.d, cfg.E, cfg.k, cfg.f, cfg.f_s
    bm = moeq4.default_block_m(T, E, k)
    stream = torch.cuda.current_stream()
    x = torch.from_numpy(synth.gen_x(cfg, T).view(np.int16)).cuda().view(torch.bfloat16)
    wr = torch.from_numpy(synth.gen_router(cfg).view(np.int16)).cuda().view(torch.bfloat16)
    W = moeq4.DeviceWeights.from_host(synth.gen_weights(cfg, 0))
    route = moeq4.RouteBuffers.alloc(T, E, k, bm)
    lg = torch.empty((T, E), dtype=torch.float32, device="cuda")
    ws = moeq4.alloc_workspace(moeq4.moe_layer_workspace_size(T, E, k, d, f, fs, bm))
    y = torch.empty((T, d), dtype=torch.bfloat16, device="cuda")
    flush = torch.empty(256 << 20, dtype=torch.uint8, device="cuda")   # larger than L2

    def timed(fn):
        for _ in range(warmup):
            fn()
        torch.cuda.synchronize()
        tot = 0.0
        for _ in range(steps):
            flush.fill_(1)
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            fn()
            e1.record(stream)
            torch.cuda.synchronize()
            tot += e0.elapsed_time(e1)
        return tot / steps

    ms_router = timed(lambda: moeq4.moe_router_topk(x, wr, route, lg, stream))
    ms_layer = timed(lambda: moeq4.moe_layer_router(x, wr, W, route, y, ws, lg, stream))
    if moeq4.moe_get_device_error(route) != 0:
        raise RuntimeError("device error word set in the router run")
    pk, _ = peaks()
    flops = 2.0 * T * E * d
    nbytes = T * d * 2 + E * d * 2 + T * E * 4 + T * k * 8
    t = ms_router * 1e-3
    bound = "tensor" if flops / (pk["bf16_tflops"] * 1e12) >= nbytes / (pk["hbm_gbs"] * 1e9) else "hbm"
    roof = {"bound": bound, "achieved_tflops": flops / t / 1e12, "achieved_gbs": nbytes / t / 1e9,
            "frac": max(flops / (pk["bf16_tflops"] * 1e12), nbytes / (pk["hbm_gbs"] * 1e9)) / t,
            "kernel": "router_topk_kernel (projection + top-k)"}
    return {"T": T, "value": T / t, "unit": UNIT, "ms_per_step": ms_router, "roofline": roof,
            "l2": "flushed (256 MB write) before every timed call",
            "layer_from_hidden_states": {"value": T / (ms_layer * 1e-3), "unit": UNIT,
                                         "ms_per_step": ms_layer},
            # the router alone, then the router + routing from its choice + the FFN
            "launches": (1 + 1 + launches_per_layer(T)) * steps}


def measure_decode(steps, warmup):
    """Small batches (decode steps) through the whole layer on the full-width
    layer (t512's widths and value recipe): T = 1, 8 and 64, each timed as
    stream launches and as replays of a captured CUDA graph, against the
    layer's HBM roofline (the touched experts' and the shared expert's 4-bit
    weights, x, y and the logits at the measured copy bandwidth)."""
    import dataclasses

    import torch

    from routing_q4_grouped_gb300 import moeq4, synth

    base = synth.CONFIGS["t512"]
    pk, _ = peaks()
    sets = [moeq4.DeviceWeights.from_host(synth.gen_weights(base, 100 + l)) for l in range(2)]
    out = {}
    launches = 0
    for T in (1, 8, 64):
        cfg = dataclasses.replace(base, T=T)
        bm = moeq4.default_block_m(T, cfg.E, cfg.k)
        xs = [torch.from_numpy(synth.gen_x(cfg, T, l).view(np.int16)).cuda().view(torch.bfloat16)
              for l in range(2)]
        ls = [torch.from_numpy(synth.gen_logits(cfg, l, T)).cuda() for l in range(2)]
        r = moeq4.RouteBuffers.alloc(T, cfg.E, cfg.k, bm)
        ws = moeq4.alloc_workspace(moeq4.moe_layer_workspace_size(T, cfg.E, cfg.k, cfg.d, cfg.f,
                                                                  cfg.f_s, bm))
        y = torch.empty((T, cfg.d), dtype=torch.bfloat16, device="cuda")
        stream = torch.cuda.Stream()
        with torch.cuda.stream(stream):
            for i in range(warmup):
                moeq4.moe_layer(xs[i % 2], ls[i % 2], sets[i % 2], r, y, ws, stream)
            stream.synchronize()
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            for i in range(steps):
                moeq4.moe_layer(xs[i % 2], ls[i % 2], sets[i % 2], r, y, ws, stream)
            e1.record(stream)
            stream.synchronize()
            ms = e0.elapsed_time(e1) / steps
            # one graph per layer set, replayed alternately
            ms_g, g_err = None, None
            try:
                graphs = []
                for l in range(2):
                    g = torch.cuda.CUDAGraph()
                    with torch.cuda.graph(g, stream=stream):
                        moeq4.moe_layer(xs[l], ls[l], sets[l], r, y, ws, stream)
                    graphs.append(g)
                for i in range(warmup):
                    graphs[i % 2].replay()
                stream.synchronize()
                e0.record(stream)
                for i in range(steps):
                    graphs[i % 2].replay()
                e1.record(stream)
                stream.synchronize()
                ms_g = e0.elapsed_time(e1) / steps
            except Exception as ex:   # capture refused: report it, keep the stream figure
                g_err = f"{type(ex).__name__}: {ex}"[:200]
                torch.cuda.synchronize()
        if moeq4.moe_get_device_error(r) != 0:
            raise RuntimeError("device error word set in the decode run")
        touched = int((r.counts.cpu().numpy() > 0).sum())
        nbytes = layer_bytes(cfg, T, touched)
        t_roof = nbytes / (pk["hbm_gbs"] * 1e9)
        out[f"T{T}"] = {
            "value": T / (ms * 1e-3), "unit": UNIT, "ms_per_step": ms,
            "graph": ({"value": T / (ms_g * 1e-3), "ms_per_step": ms_g} if ms_g else
                      {"error": g_err}),
            "path": "decode kernels" if T <= 2 else "tensor-core grouped GEMM",
            "touched_experts": touched,
            "roofline": {"bound": "hbm", "bytes": nbytes, "roofline_us": t_roof * 1e6,
                         "achieved_gbs": nbytes / (ms * 1e-3) / 1e9, "frac": t_roof / (ms * 1e-3),
                         "frac_graph": t_roof / (ms_g * 1e-3) if ms_g else None,
                         "peak_gbs": pk["hbm_gbs"]}}
        # stream launches, and the same kernels again as graph replays
        per = launches_per_layer(T, decode=T <= 2)
        launches += per * steps * (2 if ms_g else 1)
    out["launches"] = launches
    return out


def run_ours(args):
    from routing_q4_grouped_gb300 import synth

    world, rank, local = dist_setup()
    cfg = synth.CONFIGS[args.workload]
    m = measure_workload(args.workload, args, world, rank, local, args.steps, args.warmup,
                         args.sets, block_m=args.block_m)
    launches = m["launches"]
    line = {
        "metric": METRIC, "value": m["value"], "unit": UNIT, "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": m["ms_per_step"], "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic (seeded counter-based generator; random-init 4-bit weights)",
        "config": {**workload_config(cfg, args, world),
                   "l2": f"inputs larger than L2: {args.sets} layer sets of "
                         f"{m['weight_bytes'] / 1e6:.0f} MB weights cycled per step"},
        "roofline": m["roofline"],
        "layer_roofline": m["layer_roofline"],
        "grouped_gemm": m["grouped_gemm"],
        "kernels_ms": m["kernels_ms"],
        "touched_experts": m["touched_experts"],
        "e2e": m["e2e"],
        "clocks": m["clocks"],
    }
    # the other single-layer workloads, measured in the same run (same step
    # count; their own seeds, block maps and layer sets)
    if not args.no_workloads and cfg.layers == 1:
        wl = {}
        for name in ("t512", "skew", "tiny", "t4096"):
            if name == args.workload:
                continue
            o = measure_workload(name, args, world, rank, local, args.steps, args.warmup,
                                 args.sets)
            launches += o["launches"]
            wl[name] = {k2: o[k2] for k2 in ("T", "block_m", "value", "ms_per_step", "kernels_ms",
                                             "roofline", "layer_roofline", "grouped_gemm",
                                             "touched_experts", "e2e", "clocks")}
            wl[name]["unit"] = UNIT
        rt = measure_router(args.workload, args.steps, args.warmup)
        launches += rt.pop("launches")
        wl["router_" + args.workload] = rt
        dec = measure_decode(args.steps, args.warmup)
        launches += dec.pop("launches")
        wl["decode"] = dec
        line["workloads"] = wl
    line["gpu_launches"] = launches
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        b = oracle_baseline(cfg, args.block_m, steps=1)
        T = cfg.tokens_per_call
        line["cpu_baseline"] = {
            "value": T / b["sec"], "unit": UNIT, "cores": b["procs"], "kind": "oracle",
            "sample": f"one whole layer ({T} tokens, routing + every expert group + shared "
                      f"expert) over {b['procs']} host processes",
            "single_core": {"value": T / b["single_core_sec"], "unit": UNIT, "cores": 1,
                            "sample": b["single_core_note"]}}
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist

        dist.destroy_process_group()


# ------------------------------------------------------- chunked multi-layer run


def device_q4_layer(cfg, gen, device="cuda"):
    """One layer's 4-bit weights in the interchange layout, drawn on `device` from
    the seeded torch generator `gen` with the synthetic recipe (uniform codes;
    scale ~ U(0.004, 0.008) -> bf16; bias = -7.5 scale + N(0, 0.001) -> bf16).
    The chunked run holds 40 layers (18 GB); drawing them on the host takes
    minutes, and the timing does not depend on which random values they hold.
    Returns {name: tensor} with the names DeviceWeights uses."""
    import torch

    def mat(prefix, experts, rows, K):
        qw = torch.randint(0, 1 << 32, (experts, rows, K // 8), dtype=torch.int64,
                           generator=gen, device=device).to(torch.int32)   # wraps to 32 bits
        shp = (experts, rows, K // 64)
        s = (0.004 + 0.004 * torch.rand(shp, generator=gen, device=device)).to(torch.bfloat16)
        b = (-7.5 * s.float() + 0.001 * torch.randn(shp, generator=gen, device=device)).to(torch.bfloat16)
        return {prefix + "_qw": qw, prefix + "_scale": s.view(torch.int16),
                prefix + "_bias": b.view(torch.int16)}

    E, d, f, fs = cfg.E, cfg.d, cfg.f, cfg.f_s
    ts = {**mat("gu", E, 2 * f, d), **mat("dn", E, d, f)}
    if fs:
        ts.update(mat("sgu", 1, 2 * fs, d))
        ts.update(mat("sdn", 1, d, fs))
    return ts


def run_chunked(args):
    """One step = the whole chunked run: every chunk of `cfg.chunk` tokens goes
    through all `cfg.layers` layers (routing, gate/up pass, down pass, then the
    next input bf16(rms_unit(y + x))), each layer with its own weights, all
    resident in HBM. `value` = tokens of the whole run / step time."""
    import torch

    from routing_q4_grouped_gb300 import moeq4

    world, rank, local = dist_setup()
    from routing_q4_grouped_gb300 import synth

    cfg = synth.CONFIGS[args.workload]
    C, L = cfg.chunk, cfg.layers
    nch = cfg.T // C
    d, E, k, f, fs = cfg.d, cfg.E, cfg.k, cfg.f, cfg.f_s
    stream = torch.cuda.current_stream()
    gen = torch.Generator(device="cuda")
    gen.manual_seed(1_000_003 * cfg.seed + rank)
    layers = []
    for _ in range(L):
        dw = moeq4.DeviceWeights(E, d, f, fs, device_q4_layer(cfg, gen))
        dw.packed = torch.empty(moeq4.moe_q4_packed_size(E, d, f, fs), dtype=torch.uint8,
                                device="cuda")
        moeq4.moe_q4_prepack(dw, dw.packed)
        stream.synchronize()
        dw.tensors = {}
        layers.append(dw)
    x0 = torch.randn((nch, C, d), generator=gen, device="cuda").to(torch.bfloat16)
    logits = torch.randn((nch, L, C, E), generator=gen, device="cuda")   # chunk-major
    route = moeq4.RouteBuffers.alloc(C, E, k, args.block_m)
    ws = moeq4.alloc_workspace(moeq4.moe_layer_workspace_size(C, E, k, d, f, fs, args.block_m))
    y = torch.empty((C, d), dtype=torch.bfloat16, device="cuda")
    xb = [torch.empty((C, d), dtype=torch.bfloat16, device="cuda") for _ in range(2)]
    out = torch.empty((nch, C, d), dtype=torch.bfloat16, device="cuda")

    # the next layer's first gate/up weights head for L2 during this layer's
    # tail, requested from a side stream so that the request never delays the
    # main stream's next kernels
    prefetch_bytes = args.prefetch_mb << 20
    pf_stream = torch.cuda.Stream()
    pf_events = [torch.cuda.Event() for _ in range(L)]

    def run_chunk(x_in, lg, y_out):
        # layers 0..L-1 of one chunk; the last layer writes the chunk's output
        cur = x_in
        for l in range(L):
            last = l + 1 == L
            moeq4.moe_layer(cur, lg[l], layers[l], route, y_out if last else y, ws, stream)
            if prefetch_bytes:
                pf_events[l].record(stream)
                pf_stream.wait_event(pf_events[l])
                moeq4.moe_l2_prefetch(layers[(l + 1) % L].packed, prefetch_bytes, pf_stream)
            if not last:
                nxt = xb[l % 2]
                moeq4.moe_residual_rms(y, cur, nxt, stream)
                cur = nxt

    def step():
        for c in range(nch):
            run_chunk(x0[c], logits[c], out[c])

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    if moeq4.moe_get_device_error(route) != 0:
        raise RuntimeError("device error word set during warm-up")

    clocks = ClockSampler(local)
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    barrier(world)
    torch.cuda.synchronize()
    clocks.start()
    time.sleep(0.3)
    ev0.record(stream)
    for _ in range(args.steps):
        step()
    ev1.record(stream)
    torch.cuda.synchronize()
    clk = clocks.stop()
    barrier(world)
    ms_total = max_over_ranks(world, ev0.elapsed_time(ev1))
    ms_step = ms_total / args.steps
    value = cfg.T * world * args.steps / (ms_total * 1e-3)

    # gate/up kernel times over the first chunk's layers (stage events)
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(6)] for _ in range(L)]
    for row in evs:
        for e in row:
            e.record(stream)
    torch.cuda.synchronize()
    cur = x0[0]
    for l in range(L):
        moeq4.moe_debug_set_stage_events(evs[l])
        moeq4.moe_layer(cur, logits[0, l], layers[l], route, y, ws, stream)
        moeq4.moe_debug_set_stage_events([])
        if l + 1 < L:
            moeq4.moe_residual_rms(y, cur, xb[l % 2], stream)
            cur = xb[l % 2]
    torch.cuda.synchronize()
    kern = {s: statistics.mean(evs[l][j].elapsed_time(evs[l][j + 1]) for l in range(L))
            for j, s in enumerate(STAGES) if s}

    # end to end: every step copies x and all logits in from pinned host memory
    # (one copy each, on a host->device stream; chunk c waits for its inputs) and
    # every chunk's output back (device->host stream)
    x_h = x0.view(torch.int16).cpu().pin_memory()
    lg_h = logits.cpu().pin_memory()
    out_h = torch.empty((nch, C, d), dtype=torch.int16).pin_memory()
    x_d, lg_d = torch.empty_like(x0), torch.empty_like(logits)
    h2d_s, d2h_s = torch.cuda.Stream(), torch.cuda.Stream()

    def e2e_step():
        ready = []
        with torch.cuda.stream(h2d_s):
            h2d_s.wait_stream(stream)          # the previous step no longer reads x_d, lg_d
            for c in range(nch):
                x_d[c].view(torch.int16).copy_(x_h[c], non_blocking=True)
                lg_d[c].copy_(lg_h[c], non_blocking=True)
                e = torch.cuda.Event()
                e.record(h2d_s)
                ready.append(e)
        stream.wait_stream(d2h_s)              # the previous step's outputs have left `out`
        for c in range(nch):
            stream.wait_event(ready[c])
            run_chunk(x_d[c], lg_d[c], out[c])
            done = torch.cuda.Event()
            done.record(stream)
            with torch.cuda.stream(d2h_s):
                d2h_s.wait_event(done)
                out_h[c].copy_(out[c].view(torch.int16), non_blocking=True)

    e2e_step()
    torch.cuda.synchronize()
    barrier(world)
    ev0.record(stream)
    h2d_s.wait_event(ev0)
    for _ in range(args.steps):
        e2e_step()
    fin = torch.cuda.Event()
    fin.record(d2h_s)
    stream.wait_event(fin)
    ev1.record(stream)
    torch.cuda.synchronize()
    e2e_ms = max_over_ranks(world, ev0.elapsed_time(ev1))
    e2e_value = cfg.T * world * args.steps / (e2e_ms * 1e-3)
    if moeq4.moe_get_device_error(route) != 0:
        raise RuntimeError("device error word set during the timed region")

    # roofline of the dominant kernel (gate/up at T = chunk), as in the one-layer bench
    pk, pk_src = peaks()
    flops_gu = 4 * d * f * C * k + 4 * d * fs * C
    flops_dn = 2 * d * f * C * k + 2 * d * fs * C
    t_gu, t_dn = kern["gemm_gate_up_swiglu"] * 1e-3, kern["gemm_down_combine"] * 1e-3
    # the same denominator as the one-layer bench (the burst bf16 figure); the
    # sustained figure, measured under the power cap at a lower clock, is
    # reported beside it
    peak_tf = pk["bf16_tflops"]
    roof = {"bound": "tensor", "achieved": flops_gu / t_gu / 1e12, "peak": peak_tf,
            "unit": "TFLOP/s"}
    roof["frac"] = roof["achieved"] / roof["peak"]
    roof["traffic"] = None
    roof["kernel"] = "q4_grouped_gemm_kernel<0> (gate/up + SwiGLU)"
    roof["peak_source"] = f"{pk_src} (bf16 burst / hbm copy)"
    if "bf16_tflops_sustained" in pk:
        roof["sustained_peak"] = {
            "value": pk["bf16_tflops_sustained"], "unit": "TFLOP/s",
            "sm_mhz_median": pk.get("clocks_under_load", {}).get("sm_mhz_median"),
            "frac": roof["achieved"] / pk["bf16_tflops_sustained"]}
    gg_tflops = (flops_gu + flops_dn) / (t_gu + t_dn) / 1e12
    line = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms_step, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic (seeded torch generator on the device, same value recipe; random-init 4-bit weights)",
        "config": {"workload": args.workload, "T": cfg.T, "chunk": C, "layers": L, "d": d, "E": E,
                   "k": k, "f": f, "f_s": fs, "block_m": args.block_m,
                   "next_layer_prefetch_mb": args.prefetch_mb,
                   "l2": f"inputs larger than L2: {L} layers of {layers[0].nbytes / 1e6:.0f} MB weights per step",
                   "parallelism": f"replicas x{world}"},
        "roofline": roof,
        "grouped_gemm": {"tflops": gg_tflops, "frac_bf16_peak": gg_tflops / peak_tf,
                         "ms": (t_gu + t_dn) * 1e3},
        "kernels_ms": kern,
        "e2e": {"value": e2e_value, "unit": UNIT,
                "h2d_bytes_per_step": x0.numel() * 2 + logits.numel() * 4,
                "d2h_bytes_per_step": out.numel() * 2},
        "clocks": clk,
        "gpu_launches": (launches_per_layer(C) * L + (L - 1) + (L if prefetch_bytes else 0))
                        * nch * args.steps,
    }
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist

        dist.destroy_process_group()


def main():
    args = parse_args()
    from routing_q4_grouped_gb300 import synth
    cfg = synth.CONFIGS[args.workload]
    if args.block_m == "auto":
        # same rule as moeq4.default_block_m (no library load needed for the reference arm)
        args.block_m = 64 if cfg.tokens_per_call * cfg.k <= 32 * cfg.E else 128
    else:
        args.block_m = int(args.block_m)
    if args.impl == "reference":
        run_reference(args)
    elif cfg.layers > 1:
        run_chunked(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
