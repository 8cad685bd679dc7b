"""Pins for the oracle's routing: selection, weights, histogram, scan, scatter, block map."""
import json
import math
import os

import numpy as np
import pytest

import oracle as O
from routing_q4_grouped_gb300 import synth

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _brute_route(logits, k, block_m):
    """Pure-Python restatement on small inputs: sorted() selection, loops for the rest."""
    T, E = len(logits), len(logits[0])
    ids = []
    for t in range(T):
        order = sorted(range(E), key=lambda e: (-float(logits[t][e]), e))
        ids.append(order[:k])
    counts = [0] * E
    for t in range(T):
        for j in range(k):
            counts[ids[t][j]] += 1
    offsets = [0]
    for e in range(E):
        offsets.append(offsets[-1] + counts[e])
    perm = [None] * (T * k)
    fill = list(offsets[:E])
    for t in range(T):            # counting sort: visit rows in ascending (t, j)
        for j in range(k):
            e = ids[t][j]
            perm[fill[e]] = t * k + j
            fill[e] += 1
    inv = [None] * (T * k)
    for p, row in enumerate(perm):
        inv[row] = p
    tiles = []
    for e in range(E):
        s = 0
        while s < counts[e]:
            tiles.append([e, offsets[e] + s, min(block_m, counts[e] - s)])
            s += block_m
    return ids, counts, offsets, perm, inv, tiles


def test_golden_ties():
    g = json.load(open(os.path.join(GOLDEN, "route_ties.json")))
    r = O.route(np.array(g["logits"], np.float32), g["k"], g["block_m"])
    assert r.ids.tolist() == g["ids"]
    assert r.counts.tolist() == g["counts"]
    assert r.offsets.tolist() == g["offsets"]
    assert r.perm.tolist() == g["perm"]
    assert r.inv.tolist() == g["inv"]
    assert r.tiles.tolist() == g["tiles"]
    a = 1.0 / (1.0 + math.exp(-4.0))
    want = np.array([0.5, 0.5, 0.5, 0.5, a, math.exp(-4.0) * a], np.float32)
    assert np.array_equal(r.w.ravel(), want)


@pytest.mark.parametrize("seed", range(6))
def test_against_brute_force(seed):
    rng = np.random.default_rng(seed)
    T, E = int(rng.integers(1, 40)), int(rng.integers(1, 24))
    k = int(rng.integers(1, E + 1))
    bm = int(rng.integers(1, 9))
    # quantised logits so that ties are frequent
    logits = (rng.integers(-4, 5, size=(T, E)) * 0.5).astype(np.float32)
    r = O.route(logits, k, bm)
    ids, counts, offsets, perm, inv, tiles = _brute_route(logits.tolist(), k, bm)
    assert r.ids.tolist() == ids
    assert r.counts.tolist() == counts
    assert r.offsets.tolist() == offsets
    assert r.perm.tolist() == perm
    assert r.inv.tolist() == inv
    assert r.tiles.tolist() == (tiles if tiles else [])


def _check_invariants(r, logits):
    T, k, E, bm = r.T, r.k, r.E, r.block_m
    assert r.counts.sum() == T * k
    assert r.offsets[0] == 0 and r.offsets[E] == T * k
    assert np.array_equal(np.diff(r.offsets), r.counts)
    assert np.array_equal(np.sort(r.perm), np.arange(T * k))            # bijection
    assert np.array_equal(r.inv[r.perm], np.arange(T * k))              # inv . perm = id
    for t in range(T):                                                  # k distinct experts
        assert len(set(r.ids[t].tolist())) == k
    tok = r.perm // k
    for e in range(E):                                                  # group rows ascending
        grp = r.perm[r.offsets[e]:r.offsets[e + 1]]
        assert np.all(np.diff(grp) > 0)
        assert np.all(r.ids.ravel()[grp] == e)
    # each token appears exactly k times
    assert np.array_equal(np.bincount(tok, minlength=T), np.full(T, k))
    # selection: every chosen logit >= every unchosen logit of the token
    L = logits.astype(np.float64)
    chosen = np.zeros_like(L, dtype=bool)
    np.put_along_axis(chosen, r.ids.astype(np.int64), True, axis=1)
    if k < E:
        assert np.all(np.where(chosen, L, np.inf).min(1) >= np.where(chosen, -np.inf, L).max(1))
    # block map covers each row once, in order, at most block_m rows per tile
    cov = np.zeros(T * k, dtype=np.int32)
    prev_end = 0
    for e, s, n in r.tiles:
        assert 1 <= n <= bm and r.offsets[e] <= s and s + n <= r.offsets[e + 1]
        assert s == prev_end
        prev_end = s + n
        cov[s:s + n] += 1
    assert np.all(cov == 1)
    assert r.n_tiles <= O.max_tiles(T, E, k, bm)


@pytest.mark.parametrize("name,bm", [("tiny", 16), ("t512", 128), ("skew", 128), ("skew", 256)])
def test_invariants_on_workloads(name, bm):
    cfg = synth.CONFIGS[name]
    logits = synth.gen_logits(cfg)
    r = O.route(logits, cfg.k, bm)
    _check_invariants(r, logits)


def test_skew_workload_is_skewed():
    cfg = synth.CONFIGS["skew"]
    r = O.route(synth.gen_logits(cfg), cfg.k, 128)
    assert (r.counts == 0).sum() >= 24                       # dozens of empty experts
    assert (r.counts > 0.10 * cfg.T * cfg.k).sum() >= 2      # a few hold >10% of rows


def test_weights_closed_form():
    cfg = synth.CONFIGS["t512"]
    logits = synth.gen_logits(cfg)[:200]
    r = O.route(logits, cfg.k, 128)
    L = logits.astype(np.float64)
    sel = np.take_along_axis(L, r.ids.astype(np.int64), 1)
    # renormalised top-k softmax equals exp(l - l_max) / sum over the chosen only
    ref = np.exp(sel - sel[:, :1]) / np.exp(sel - sel[:, :1]).sum(1, keepdims=True)
    assert np.array_equal(r.w, ref.astype(np.float32))
    assert np.all(np.abs(r.w.astype(np.float64).sum(1) - 1.0) <= cfg.k * 2.0 ** -24)
    assert np.all(np.diff(r.w, axis=1) <= 0)                 # descending with the logits


def test_equal_logits_k_equals_E():
    r = O.route(np.zeros((5, 8), np.float32), 8, 4)
    assert np.all(r.w == np.float32(0.125))
    assert r.ids.tolist() == [list(range(8))] * 5


def test_nan_rejected():
    logits = np.zeros((2, 4), np.float32)
    logits[1, 2] = np.nan
    with pytest.raises(ValueError):
        O.route(logits, 2)


def test_single_expert_and_single_token():
    r = O.route(np.array([[0.3]], np.float32), 1, 128)
    assert r.ids.tolist() == [[0]] and r.w.tolist() == [[1.0]]
    assert r.tiles.tolist() == [[0, 0, 1]]


# ------------------------------------------------------------ router projection


def test_router_logits_one_hot_rows_pick_columns():
    # Wr[e] = unit vector at column c_e: the logit is that column of x, exactly
    cfg = synth.CONFIGS["tiny"]
    x = synth.gen_x(cfg, 16)
    cols = np.array([3, 0, 255, 17, 17, 100, 1, 64])
    wr = np.zeros((8, cfg.d), np.uint16)
    wr[np.arange(8), cols] = 0x3F80                      # bf16 1.0
    got = O.router_logits(x, wr)
    assert np.array_equal(got, O.bf16_value(x)[:, cols])


def test_router_logits_constant_rows_are_scaled_row_sums():
    import math
    cfg = synth.CONFIGS["tiny"]
    x = synth.gen_x(cfg, 12)
    consts = [0.5, -2.0, 0.0078125, 3.0]
    wr = np.stack([np.full(cfg.d, O.to_bf16(c), np.uint16) for c in consts])
    got = O.router_logits(x, wr)
    xv = O.bf16_value(x)
    for t in range(12):
        s = math.fsum(float(v) for v in xv[t])
        for e, c in enumerate(consts):
            assert abs(got[t, e] - c * s) <= 1e-12 * max(1.0, abs(c * s))


def test_router_logits_brute_force_loops():
    rng = np.random.default_rng(4)
    x = O.to_bf16(rng.standard_normal((3, 8)))
    wr = O.to_bf16(rng.standard_normal((4, 8)))
    xv, wv = O.bf16_value(x), O.bf16_value(wr)
    got = O.router_logits(x, wr)
    for t in range(3):
        for e in range(4):
            acc = 0.0
            for c in range(8):
                acc += float(xv[t, c]) * float(wv[e, c])
            assert abs(got[t, e] - acc) <= 1e-12


def test_router_weights_give_unit_scale_logits():
    cfg = synth.CONFIGS["t512"]
    lg = O.router_logits(synth.gen_x(cfg, 256), synth.gen_router(cfg))
    assert 0.9 < lg.std() < 1.1 and abs(lg.mean()) < 0.05
