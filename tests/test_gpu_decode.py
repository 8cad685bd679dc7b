"""The small-batch (decode) expert FFN against the oracle within the layer
tolerance, on the full-width layer (d = 2048, 256 experts, top-8, shared
expert) at T = 1, 8 and 64, with ragged and empty expert groups, and the
automatic choice between the decode path and the tensor-core grouped GEMM."""
import dataclasses

import numpy as np
import pytest
import torch

import oracle as O
from routing_q4_grouped_gb300 import moeq4, synth
from gpu_helpers import assert_route_equal, assert_y_close, bits, dev, route_np

pytestmark = pytest.mark.gpu


def _setup(cfg, T, layer=0, bm=64):
    W = synth.gen_weights(cfg, layer)
    x = synth.gen_x(cfg, T, layer)
    logits = synth.gen_logits(cfg, layer, T)
    DW = moeq4.DeviceWeights.from_host(W)
    r = moeq4.RouteBuffers.alloc(T, cfg.E, cfg.k, bm)
    ws = moeq4.alloc_workspace(moeq4.moe_layer_workspace_size(T, cfg.E, cfg.k, cfg.d, cfg.f,
                                                              cfg.f_s, bm))
    return W, x, logits, DW, r, ws


@pytest.mark.parametrize("T", [1, 8, 64])
def test_decode_path_matches_oracle(T):
    cfg = synth.CONFIGS["t512"]
    W, x, logits, DW, r, ws = _setup(cfg, T, layer=T)
    rsz = (moeq4.moe_route_workspace_size(T, cfg.E, cfg.k) + 255) // 256 * 256
    moeq4.moe_route(dev(logits), r, ws[:rsz])
    y = torch.empty((T, cfg.d), dtype=torch.bfloat16, device="cuda")
    moeq4.moe_expert_ffn_decode(dev(x), DW, r, y, ws[rsz:])
    assert moeq4.moe_get_device_error(r) == 0
    ref_r = O.route(logits, cfg.k, 64)
    assert_route_equal(route_np(r), ref_r)
    assert_y_close(bits(y), O.expert_ffn(x, W, ref_r))


def test_decode_without_shared_expert_and_block_map_of_one_row_tiles():
    cfg = dataclasses.replace(synth.CONFIGS["t512"], f_s=0)
    T = 12
    W, x, logits, DW, r, ws = _setup(cfg, T, bm=1)      # one tile per routed row
    rsz = (moeq4.moe_route_workspace_size(T, cfg.E, cfg.k) + 255) // 256 * 256
    moeq4.moe_route(dev(logits), r, ws[:rsz])
    y = torch.empty((T, cfg.d), dtype=torch.bfloat16, device="cuda")
    moeq4.moe_expert_ffn_decode(dev(x), DW, r, y, ws[rsz:])
    assert moeq4.moe_get_device_error(r) == 0
    assert_y_close(bits(y), O.expert_ffn(x, W, O.route(logits, cfg.k, 1)))


@pytest.mark.parametrize("T", [16, 64])
def test_layer_switches_paths_on_one_workspace(T):
    # the same batch size through the decode path, the tensor-core path and the
    # decode path again on one workspace: neither path may depend on state the
    # other leaves behind
    cfg = synth.CONFIGS["t512"]
    W = synth.gen_weights(cfg, 3)
    DW = moeq4.DeviceWeights.from_host(W)
    ws = moeq4.alloc_workspace(moeq4.moe_layer_workspace_size(T, cfg.E, cfg.k, cfg.d, cfg.f,
                                                              cfg.f_s, 64))
    r = moeq4.RouteBuffers.alloc(T, cfg.E, cfg.k, 64)
    y = torch.empty((T, cfg.d), dtype=torch.bfloat16, device="cuda")
    try:
        for i, dmax in enumerate((64, 0, 64, 0)):
            moeq4.moe_debug_set_decode_max_t(dmax)
            x = synth.gen_x(cfg, T, 7 + i)
            logits = synth.gen_logits(cfg, 7 + i, T)
            moeq4.moe_layer(dev(x), dev(logits), DW, r, y, ws)
            assert moeq4.moe_get_device_error(r) == 0
            assert_y_close(bits(y), O.expert_ffn(x, W, O.route(logits, cfg.k, 64)))
    finally:
        moeq4.moe_debug_set_decode_max_t(2)


def test_decode_rejects_large_batches():
    cfg = synth.CONFIGS["t512"]
    T = 65
    W, x, logits, DW, r, ws = _setup(cfg, T)
    y = torch.empty((T, cfg.d), dtype=torch.bfloat16, device="cuda")
    with pytest.raises(moeq4.MoeError):
        moeq4.moe_expert_ffn_decode(dev(x), DW, r, y, ws)
