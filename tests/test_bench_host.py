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
