"""The fused router (projection + top-k on the tensor cores) against the oracle.

The logits come from an fp32 accumulation on the GPU and a float64 one in the
oracle, so they are compared within the accumulation's error bound. The choice
of experts is an integer decision taken on floating point: the oracle takes it
on the GPU's own fp32 logits (same precision, same values), and ids, weights and
the whole routing result must then match bit for bit. Where the oracle's own
logits leave a clear margin between the k-th and the next expert, the two
choices must also agree.
"""
import dataclasses

import numpy as np
import pytest
import torch

import oracle as O
from routing_q4_grouped_gb300 import moeq4, synth
from gpu_helpers import assert_route_equal, assert_y_close, bits, dev, route_np

pytestmark = pytest.mark.gpu


def _router_gpu(x, wr, k, block_m=128):
    T, E = x.shape[0], wr.shape[0]
    out = moeq4.RouteBuffers.alloc(T, E, k, block_m)
    logits = torch.empty((T, E), dtype=torch.float32, device="cuda")
    moeq4.moe_router_topk(dev(x), dev(wr), out, logits)
    err = moeq4.moe_get_device_error(out)
    return out, logits.cpu().numpy(), err


def _check_logits(got, x, wr):
    ref = O.router_logits(x, wr)
    # fp32 accumulation of exact bf16 products over d terms: |error| <= d * 2^-24 * sum |x_i w_i|
    mag = np.abs(O.bf16_value(x)) @ np.abs(O.bf16_value(wr)).T
    d = x.shape[1]
    assert np.all(np.abs(got - ref) <= d * 2.0 ** -24 * mag + 1e-30)
    return ref, d * 2.0 ** -24 * mag


@pytest.mark.parametrize("name,T", [("t4096", 4096), ("t512", 512), ("t512", 300), ("t512", 1)])
def test_router_logits_topk_and_weights(name, T):
    cfg = synth.CONFIGS[name]
    x = synth.gen_x(cfg, T)
    wr = synth.gen_router(cfg)
    out, lg, err = _router_gpu(x, wr, cfg.k)
    assert err == 0
    ref, bound = _check_logits(lg, x, wr)
    # the choice and weights, taken by the oracle on the GPU's fp32 logits
    r = O.route(lg, cfg.k, 128)
    g = route_np(out)
    assert np.array_equal(g["ids"], r.ids)
    assert np.array_equal(g["w"].view(np.uint32), r.w.view(np.uint32))
    # and on the oracle's own logits where the margin exceeds both error bounds
    r64 = O.route(ref.astype(np.float32), cfg.k, 128)
    srt = -np.sort(-ref, axis=1)
    margin = srt[:, cfg.k - 1] - srt[:, cfg.k]
    clear = margin > 4 * bound.max(axis=1) + 1e-6
    assert clear.mean() > 0.5          # the worst-case bound is loose; most tokens still qualify
    assert np.array_equal(np.sort(g["ids"][clear], axis=1), np.sort(r64.ids[clear], axis=1))


def test_router_small_expert_counts_and_ties():
    # E = 16 (the smallest MMA width), k = 1 and k = 8; duplicated router rows
    # give equal logits: the lower expert index must win
    cfg = dataclasses.replace(synth.CONFIGS["tiny"], E=16, d=256)
    x = synth.gen_x(cfg, 200)
    wr = synth.gen_router(cfg)
    wr[5] = wr[2]
    wr[9] = wr[2]
    for k in (1, 8):
        out, lg, err = _router_gpu(x, wr, k)
        assert err == 0
        _check_logits(lg, x, wr)
        assert np.array_equal(lg[:, 5], lg[:, 2]) and np.array_equal(lg[:, 9], lg[:, 2])
        r = O.route(lg, k, 128)
        g = route_np(out)
        assert np.array_equal(g["ids"], r.ids)
        assert np.array_equal(g["w"].view(np.uint32), r.w.view(np.uint32))


@pytest.mark.parametrize("E", [128, 160, 240, 256])
def test_router_expert_halves_and_cross_half_ties(E):
    # E = 160 and 256 split the experts over a cluster of two CTAs (80 / 128
    # each); 128 and 240 run one CTA per token tile (6 and 4 ring stages). Router
    # rows copied across the halves give equal logits in both CTAs: the lower
    # expert index must still come first.
    cfg = dataclasses.replace(synth.CONFIGS["t512"], E=E)
    x = synth.gen_x(cfg, 300)
    wr = synth.gen_router(cfg)
    wr[E - 1] = wr[0]
    wr[E // 2] = wr[1]
    wr[E // 2 + 3] = wr[E // 2 - 2]
    out, lg, err = _router_gpu(x, wr, cfg.k)
    assert err == 0
    _check_logits(lg, x, wr)
    assert np.array_equal(lg[:, E - 1], lg[:, 0]) and np.array_equal(lg[:, E // 2], lg[:, 1])
    r = O.route(lg, cfg.k, 128)
    g = route_np(out)
    assert np.array_equal(g["ids"], r.ids)
    assert np.array_equal(g["w"].view(np.uint32), r.w.view(np.uint32))
    # the copies make some tokens choose a duplicated pair: both members, lower first
    both = np.isin(r.ids, [0]).any(axis=1) & np.isin(r.ids, [E - 1]).any(axis=1)
    for t in np.nonzero(both)[0]:
        row = list(r.ids[t])
        assert row.index(0) < row.index(E - 1)


@pytest.mark.parametrize("k", [1, 2, 6])
def test_router_clusters_with_fewer_choices(k):
    # E = 256: four CTAs per token tile, each keeping its best k of 64 experts;
    # the merged lists must still give the k largest of all 256
    cfg = synth.CONFIGS["t512"]
    x = synth.gen_x(cfg, 200)
    wr = synth.gen_router(cfg)
    out, lg, err = _router_gpu(x, wr, k)
    assert err == 0
    _check_logits(lg, x, wr)
    r = O.route(lg, k, 128)
    g = route_np(out)
    assert np.array_equal(g["ids"], r.ids)
    assert np.array_equal(g["w"].view(np.uint32), r.w.view(np.uint32))


@pytest.mark.parametrize("name,T", [("t4096", 4096), ("skew", 2048)])
def test_routing_from_router_ids(name, T):
    cfg = synth.CONFIGS[name]
    x = synth.gen_x(cfg, T)
    wr = synth.gen_router(cfg)
    out, lg, err = _router_gpu(x, wr, cfg.k)
    ws = moeq4.alloc_workspace(moeq4.moe_route_workspace_size(T, cfg.E, cfg.k))
    moeq4.moe_route_ids(out, ws)
    assert moeq4.moe_get_device_error(out) == 0
    assert_route_equal(route_np(out), O.route(lg, cfg.k, 128))


def test_layer_from_hidden_states():
    cfg = synth.CONFIGS["t512"]
    T = cfg.T
    W = synth.gen_weights(cfg)
    x = synth.gen_x(cfg, T)
    wr = synth.gen_router(cfg)
    DW = moeq4.DeviceWeights.from_host(W)
    r = moeq4.RouteBuffers.alloc(T, cfg.E, cfg.k, 64)
    ws = moeq4.alloc_workspace(moeq4.moe_layer_workspace_size(T, cfg.E, cfg.k, cfg.d, cfg.f,
                                                              cfg.f_s, 64))
    y = torch.empty((T, cfg.d), dtype=torch.bfloat16, device="cuda")
    lg = torch.empty((T, cfg.E), dtype=torch.float32, device="cuda")
    moeq4.moe_layer_router(dev(x), dev(wr), DW, r, y, ws, lg)
    assert moeq4.moe_get_device_error(r) == 0
    lgh = lg.cpu().numpy()
    _check_logits(lgh, x, wr)
    ref_r = O.route(lgh, cfg.k, 64)
    assert_route_equal(route_np(r), ref_r)
    assert_y_close(bits(y), O.expert_ffn(x, W, ref_r))


def test_router_rejects_unsupported_shapes():
    cfg = synth.CONFIGS["t512"]
    x = dev(synth.gen_x(cfg, 8))
    wr = dev(synth.gen_router(cfg))
    out = moeq4.RouteBuffers.alloc(8, cfg.E, 9, 128)        # k above the fused router's 8
    with pytest.raises(moeq4.MoeError):
        moeq4.moe_router_topk(x, wr, out)
    out = moeq4.RouteBuffers.alloc(8, 250, 8, 128)           # E not a multiple of 16
    with pytest.raises(moeq4.MoeError):
        moeq4.moe_router_topk(x, wr[:250].contiguous(), out)
