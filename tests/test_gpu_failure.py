"""Failure detection on the GPU without a fault, trap or hang.

A routing call whose block-ticket counter was left dirty (1 instead of 0)
hands out ids 1..nblk: the block that draws nblk refuses it (out of range), so
the grid barrier never fills, and no block has id 0, so the decoupled-lookback
waits never find an inclusive prefix. Both waits run out after the configured
limit, the kernel returns, and the error word carries MOE_DEVERR_BAD_WORKSPACE
and MOE_DEVERR_SCAN_TIMEOUT; the scatter's own checks keep every write inside
its buffer. The wait limit is read once per process, so the call runs in a
child process with MOEQ4_WAIT_TIMEOUT_MS=100.
"""
import os
import subprocess
import sys

import pytest

from routing_q4_grouped_gb300 import moeq4

pytestmark = pytest.mark.gpu

CHILD = r'''
import time
import torch
from routing_q4_grouped_gb300 import moeq4, synth
cfg = synth.CONFIGS["t512"]
lg = torch.from_numpy(synth.gen_logits(cfg)).cuda()
T, E = lg.shape
out = moeq4.RouteBuffers.alloc(T, E, cfg.k, 128)
ws = moeq4.alloc_workspace(moeq4.moe_route_workspace_size(T, E, cfg.k))
ws[0:4].view(torch.int32)[0] = 1                 # the ticket counter opens the workspace
torch.cuda.synchronize()
t0 = time.time()
moeq4.moe_route(lg, out, ws)
err = moeq4.moe_get_device_error(out)
print("ERR", err, "SECONDS", time.time() - t0)
'''


def test_dirty_routing_scratch_times_out_and_reports():
    env = dict(os.environ, MOEQ4_WAIT_TIMEOUT_MS="100")
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    r = subprocess.run([sys.executable, "-c", CHILD], env=env, cwd=root, capture_output=True,
                       text=True, timeout=600)
    assert r.returncode == 0, r.stderr[-3000:]
    line = [ln for ln in r.stdout.splitlines() if ln.startswith("ERR")][-1].split()
    err, secs = int(line[1]), float(line[3])
    assert err & moeq4.MOE_DEVERR_BAD_WORKSPACE
    assert err & moeq4.MOE_DEVERR_SCAN_TIMEOUT
    assert secs < 30   # bounded by the 100 ms wait limit, not a hang
