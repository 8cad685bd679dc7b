"""Runs the oracle's expert groups of one layer in several host processes.

TEST INFRASTRUCTURE ONLY, like the rest of ``oracle/``: the benchmark uses it
to time the oracle, as it stands, on whole layers over the host cores. It adds
no arithmetic: every worker calls :func:`oracle.expert_ffn` on some expert
groups and returns its weighted partial sum; the parent adds the partial sums
(float64) and rounds y to bf16 once. Workers are spawned (a forked child of a
process that has used a GPU can hang) and keep the layer's arrays as
memory-mapped ``.npy`` files.
"""
from __future__ import annotations

import os
import queue
import tempfile
import time

import numpy as np

_WEIGHT_FIELDS = ("gu_qw", "gu_scale", "gu_bias", "dn_qw", "dn_scale", "dn_bias",
                  "sgu_qw", "sgu_scale", "sgu_bias", "sdn_qw", "sdn_scale", "sdn_bias")


def _worker(wid, data_dir, control, groups, done):
    import oracle as O
    from routing_q4_grouped_gb300 import synth

    x = W = None
    acc = None
    while True:
        msg = control.get()
        if msg is None:
            return
        if msg[0] == "load":
            meta = msg[1]
            arr = {n: np.load(os.path.join(data_dir, n + ".npy"), mmap_mode="r")
                   for n in meta["names"]}
            x = arr.pop("x")
            W = synth.Q4Weights(meta["E"], meta["d"], meta["f"], meta["f_s"], **arr)
            done.put(("loaded", wid, True))
        elif msg[0] == "step":
            r, out_path = msg[1], msg[2]
            if acc is None or acc.shape != x.shape:
                acc = np.zeros(x.shape, dtype=np.float64)
            else:
                acc.fill(0.0)
            used = False
            while True:
                g = groups.get()
                if g is None:
                    break
                experts, shared = g
                # the rows of this group's tokens only (every token is independent)
                if shared:
                    tok = np.arange(x.shape[0])
                else:
                    rows = np.concatenate([r.perm[r.offsets[e]:r.offsets[e + 1]] for e in experts])
                    tok = np.unique(rows // r.k)
                _, a = O.expert_ffn(x, W, r, tokens=tok, experts=experts, shared=shared,
                                    return_acc=True)
                acc[tok] += a
                used = True
            if used:
                np.save(out_path, acc)
            done.put(("step", wid, used))


class OraclePool:
    """`procs` worker processes that run the oracle's expert groups of one layer."""

    def __init__(self, procs: int):
        import multiprocessing as mp

        ctx = mp.get_context("spawn")
        self.procs = procs
        self.dir = tempfile.mkdtemp(prefix="oracle_pool_")
        self.control = [ctx.Queue() for _ in range(procs)]
        self.groups = ctx.Queue()
        self.done = ctx.Queue()
        self.workers = [ctx.Process(target=_worker, daemon=True,
                                    args=(i, self.dir, self.control[i], self.groups, self.done))
                        for i in range(procs)]
        for w in self.workers:
            w.start()

    def _collect(self, n, timeout):
        """n messages from the workers; raises if a worker died or time ran out."""
        out, t_end = [], time.time() + timeout
        while len(out) < n:
            try:
                out.append(self.done.get(timeout=1.0))
            except queue.Empty:
                dead = [w.exitcode for w in self.workers if not w.is_alive()]
                if dead:
                    raise RuntimeError(f"oracle worker exited with codes {dead}")
                if time.time() > t_end:
                    raise TimeoutError("oracle workers did not answer")
        return out

    def load(self, W, x):
        names = ["x"]
        np.save(os.path.join(self.dir, "x.npy"), np.asarray(x))
        for f in _WEIGHT_FIELDS:
            a = getattr(W, f)
            if a is not None:
                np.save(os.path.join(self.dir, f + ".npy"), a)
                names.append(f)
        meta = {"names": names, "E": W.E, "d": W.d, "f": W.f, "f_s": W.f_s}
        for q in self.control:
            q.put(("load", meta))
        self._collect(self.procs, 900)
        self.f_s, self.shape = W.f_s, np.asarray(x).shape

    def layer(self, logits, k, block_m):
        """One layer: routing in this process, the expert groups over the
        workers (largest first, one group per task, the shared expert as a task
        of its own), partial sums added. Returns (Route, y bf16 bits)."""
        import oracle as O

        r = O.route(logits, k, block_m)
        paths = [os.path.join(self.dir, f"acc{i}.npy") for i in range(self.procs)]
        for i, q in enumerate(self.control):
            q.put(("step", r, paths[i]))
        if self.f_s:
            self.groups.put(([], True))
        for e in np.argsort(-r.counts, kind="stable"):
            if r.counts[e] > 0:
                self.groups.put(([int(e)], False))
        for _ in range(self.procs):
            self.groups.put(None)
        acc = np.zeros(self.shape, dtype=np.float64)
        for msg in self._collect(self.procs, 3600):
            if msg[2]:
                acc += np.load(paths[msg[1]])
        return r, O.to_bf16(acc)

    def close(self):
        for q in self.control:
            q.put(None)
        for w in self.workers:
            w.join(timeout=30)
            if w.is_alive():
                w.terminate()
        for n in os.listdir(self.dir):
            os.unlink(os.path.join(self.dir, n))
        os.rmdir(self.dir)
