"""GPU routing against the oracle: every routing output (ids, weights, counts,
offsets, permutation, inverse, block map) bit-exact, on the workloads and the
edge cases."""
import numpy as np
import pytest
import torch

import oracle as O
from routing_q4_grouped_gb300 import moeq4, synth
from gpu_helpers import assert_route_equal, route_gpu, route_np

pytestmark = pytest.mark.gpu


def _check(logits, k, bm, ws=None):
    out, err, ws = route_gpu(logits, k, bm, ws)
    assert err == 0
    g = route_np(out)
    r = O.route(logits, k, bm)
    assert_route_equal(g, r)
    return g, ws


@pytest.mark.parametrize("name,bm", [("tiny", 16), ("tiny", 128), ("t512", 128), ("t4096", 128),
                                     ("t4096", 64), ("skew", 128), ("skew", 32)])
def test_workloads(name, bm):
    cfg = synth.CONFIGS[name]
    _check(synth.gen_logits(cfg), cfg.k, bm)


def test_chunked_first_chunk_of_each_of_three_layers():
    cfg = synth.CONFIGS["chunked"]
    for layer in range(3):
        logits = synth.gen_logits(cfg, layer=layer, T=cfg.chunk)
        _check(logits, cfg.k, 128)


@pytest.mark.parametrize("T,E,k", [(1, 256, 8), (33, 256, 8), (31, 8, 2), (7, 1, 1), (16, 8, 8),
                                   (100, 40, 5), (65, 1000, 32), (257, 64, 3), (2, 1024, 1)])
def test_shapes_and_ragged_blocks(T, E, k):
    rng = np.random.default_rng(T * 7 + E)
    logits = rng.standard_normal((T, E)).astype(np.float32)
    _check(logits, k, 16)


@pytest.mark.parametrize("T,E,k", [(6000, 1024, 8), (40000, 256, 8), (100000, 256, 8)])
def test_large_grids(T, E, k):
    # many tokens per block; at T = 100000 the block's shared memory caps the
    # tokens per block, so the grid grows past 128 blocks (266)
    rng = np.random.default_rng(T + E)
    logits = rng.standard_normal((T, E)).astype(np.float32)
    _check(logits, k, 128)


def test_ties_and_equal_logits():
    rng = np.random.default_rng(3)
    logits = (rng.integers(-2, 3, size=(300, 64)) * 0.25).astype(np.float32)
    _check(logits, 6, 8)
    _check(np.zeros((40, 32), np.float32), 32, 128)


def test_empty_input():
    out, err, _ = route_gpu(np.zeros((0, 16), np.float32), 2, 128)
    assert err == 0
    assert out.counts.cpu().numpy().tolist() == [0] * 16
    assert out.offsets.cpu().numpy().tolist() == [0] * 17
    assert int(out.n_tiles[0]) == 0


def test_workspace_left_clean_and_reusable():
    cfg = synth.CONFIGS["t512"]
    logits = synth.gen_logits(cfg)
    g1, ws = _check(logits, cfg.k, 128)
    g2, _ = _check(synth.gen_logits(synth.CONFIGS["t4096"])[:512], cfg.k, 128, ws)
    g3, _ = _check(logits, cfg.k, 128, ws)
    for key in ("ids", "perm", "inv", "tiles"):
        assert np.array_equal(g1[key], g3[key])


def test_workspace_contents_do_not_matter():
    # the count rows may hold anything at launch: the choosing launch writes
    # every row before the placing launch reads it
    cfg = synth.CONFIGS["t512"]
    logits = synth.gen_logits(cfg)
    g1, ws = _check(logits, cfg.k, 128)
    ws.view(torch.int32).fill_(12345)
    g2, _ = _check(logits, cfg.k, 128, ws)
    ws.view(torch.int32).fill_(-1)
    g3, _ = _check(logits, cfg.k, 128, ws)
    for key in ("ids", "w", "perm", "inv", "tiles"):
        assert np.array_equal(g1[key], g2[key]) and np.array_equal(g1[key], g3[key])


def test_nonfinite_logit_sets_device_error():
    logits = np.random.default_rng(0).standard_normal((64, 16)).astype(np.float32)
    logits[5, 3] = np.nan
    out, err, _ = route_gpu(logits, 2, 128)
    assert err & moeq4.MOE_DEVERR_NONFINITE_LOGIT
    # the other tokens are still routed exactly
    g = route_np(out)
    ref = O.route(np.delete(logits, 5, axis=0), 2, 128)
    assert np.array_equal(np.delete(g["ids"], 5, axis=0), ref.ids)
