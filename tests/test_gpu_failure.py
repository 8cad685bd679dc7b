"""Failure detection on the GPU without a fault, trap or hang.

The down pass of the expert FFN ends with a grid barrier (one CTA per
multiprocessor) whose arrival counter, at the start of the FFN workspace, must
be zero at launch. Two dirty counters, each in a call of its own:

* left at -1: no CTA ever sees the count reach the grid size, so every CTA's
  wait runs out after the configured limit; the kernel reports
  MOE_DEVERR_PIPE_TIMEOUT, skips the bf16 conversion and returns;
* left at a value above the grid size: the CTAs see it at arrival, report
  MOE_DEVERR_BAD_WORKSPACE and do not wait at all.

Routing itself has no cross-block waits (two launches chained on the stream),
so its workspace contents cannot make it wait. The wait limit is read once per
process, so the calls run in a child process with MOEQ4_WAIT_TIMEOUT_MS=100.
"""
import os
import subprocess
import sys

import pytest

from routing_q4_grouped_gb300 import moeq4

pytestmark = pytest.mark.gpu

CHILD = r'''
import time
import numpy as np
import torch
from routing_q4_grouped_gb300 import moeq4, synth
cfg = synth.CONFIGS["tiny"]
W = moeq4.DeviceWeights.from_host(synth.gen_weights(cfg))
x = torch.from_numpy(synth.gen_x(cfg).view(np.int16)).cuda().view(torch.bfloat16)
lg = torch.from_numpy(synth.gen_logits(cfg)).cuda()
T, E = lg.shape
for start in (-1, 1 << 20):
    r = moeq4.RouteBuffers.alloc(T, E, cfg.k, 128)
    rws = moeq4.alloc_workspace(moeq4.moe_route_workspace_size(T, E, cfg.k))
    moeq4.moe_route(lg, r, rws)
    fws = moeq4.alloc_workspace(moeq4.moe_ffn_workspace_size(T, E, cfg.k, cfg.d, cfg.f, cfg.f_s))
    fws[0:4].view(torch.int32)[0] = start       # arrival counter of the down pass's grid barrier
    y = torch.empty_like(x)
    torch.cuda.synchronize()
    t0 = time.time()
    moeq4.moe_expert_ffn(x, W, r, y, fws)
    err = moeq4.moe_get_device_error(r)
    print("ERR", start, err, "SECONDS", time.time() - t0)
'''


def test_dirty_ffn_barrier_counter_times_out_and_reports():
    env = dict(os.environ, MOEQ4_WAIT_TIMEOUT_MS="100")
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    r = subprocess.run([sys.executable, "-c", CHILD], env=env, cwd=root, capture_output=True,
                       text=True, timeout=600)
    assert r.returncode == 0, r.stderr[-3000:]
    res = {}
    for ln in r.stdout.splitlines():
        if ln.startswith("ERR"):
            f = ln.split()
            res[int(f[1])] = (int(f[2]), float(f[4]))
    err, secs = res[-1]
    assert err & moeq4.MOE_DEVERR_PIPE_TIMEOUT
    assert secs < 30   # bounded by the 100 ms wait limit, not a hang
    err, secs = res[1 << 20]
    assert err & moeq4.MOE_DEVERR_BAD_WORKSPACE
    assert not err & moeq4.MOE_DEVERR_PIPE_TIMEOUT
    assert secs < 30
