"""Failure detection on the GPU without a fault, trap or hang.

A routing call whose scratch counters were left dirty makes half of the
selection blocks refuse their (out-of-range) block ids and leaves the others'
decoupled-lookback waits without predecessors: those waits run out after the
configured limit, every kernel returns, and the error word carries both
MOE_DEVERR_BAD_WORKSPACE and MOE_DEVERR_SCAN_TIMEOUT. The scatter kernel's own
checks keep every write inside its buffer. The wait limit is read once per
process, so the call runs in a child process with MOEQ4_WAIT_TIMEOUT_MS=100.
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
nblk = (T + 31) // 32
ctr = (4 * nblk * E + 255) // 256 * 256          # the counters follow the lookback words
ws[ctr:ctr + 4].view(torch.int32)[0] = nblk // 2  # ticket counter left dirty
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
