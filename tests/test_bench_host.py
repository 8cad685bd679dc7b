"""Host logic of bench.py that needs no GPU: the traffic figure is taken from a
committed ncu summary only while the kernel sources are the ones it was
captured on, and the per-rank synthetic layers are disjoint."""
import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402


def test_traffic_follows_the_kernel_source_hash(monkeypatch):
    for wl in ("t4096", "t512"):
        t = bench.profiled_traffic(wl)
        assert t is None or t > 0
        if t is not None:
            # a summary taken on other sources is not used
            monkeypatch.setattr(bench, "kernel_source_hash", lambda: "0" * 16)
            assert bench.profiled_traffic(wl) is None
            monkeypatch.undo()
    assert bench.profiled_traffic("no_such_workload") is None


def test_layer_ids_disjoint_per_rank():
    ids = [bench.layer_ids(r, 3) for r in range(4)]
    flat = [i for x in ids for i in x]
    assert len(flat) == len(set(flat)) == 12


def test_device_weight_recipe_on_the_host():
    # the chunked run draws its 40 layers with torch; same shapes, types and value recipe
    import dataclasses

    import torch

    from routing_q4_grouped_gb300 import synth

    cfg = dataclasses.replace(synth.CONFIGS["chunked"], E=4, d=256, f=128, f_s=128)
    g = torch.Generator(device="cpu")
    g.manual_seed(5)
    ts = bench.device_q4_layer(cfg, g, device="cpu")
    W = synth.gen_weights(cfg, 0)
    for n, t in ts.items():
        ref = getattr(W, n)
        assert tuple(t.shape) == ref.shape, n
        assert t.element_size() == ref.dtype.itemsize, n
    s = ts["gu_scale"].view(torch.bfloat16).float()
    b = ts["gu_bias"].view(torch.bfloat16).float()
    assert s.min() >= 0.004 - 1e-5 and s.max() <= 0.008 + 1e-5
    assert (b + 7.5 * s).abs().max() < 0.006          # bias = -7.5 s + N(0, 0.001)
    q = ts["gu_qw"]
    nib = torch.stack([(q >> (4 * i)) & 15 for i in range(8)]).flatten()
    assert nib.min() == 0 and nib.max() == 15
    assert abs(nib.float().mean().item() - 7.5) < 0.1  # uniform codes


def test_launch_count_follows_the_routing_block_rule():
    # routing is one launch while one block (kRouteTokensMin tokens at least)
    # covers the batch, two otherwise; the FFN adds two launches, or three on
    # the small-batch path
    import re
    src = open(os.path.join(ROOT, "routing_q4_grouped_gb300", "csrc", "internal.h")).read()
    tmin = int(re.search(r"kRouteTokensMin\s*=\s*(\d+)", src).group(1))
    assert bench.launches_per_layer(1) == 1 + 2
    assert bench.launches_per_layer(tmin) == 1 + 2
    assert bench.launches_per_layer(tmin + 1) == 2 + 2
    assert bench.launches_per_layer(4096) == 4
    assert bench.launches_per_layer(1, decode=True) == 1 + 3
