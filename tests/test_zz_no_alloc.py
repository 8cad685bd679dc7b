"""moe_route_noalloc: routing for callers that cannot allocate device memory.

Such callers (a serving process that hands out fixed arenas, a plugin without
access to its host framework's allocator) get moe_route with the library's own
fixed scratch array instead of a caller workspace. These checks run it through
the C-ABI and compare it with moe_route, which takes a caller workspace, on two
calls in a row: the routing outputs must be identical (the routing tests
require bit-exact results), including on the second call, which reuses the
scratch the first call left behind.
"""
import numpy as np
import pytest
import torch

from routing_q4_grouped_gb300 import moeq4, synth

pytestmark = pytest.mark.gpu

FIELDS = ("ids", "w", "counts", "offsets", "perm", "inv")


def _route_ws(logits, k, bm):
    T, E = logits.shape
    out = moeq4.RouteBuffers.alloc(T, E, k, bm)
    ws = moeq4.alloc_workspace(moeq4.moe_route_workspace_size(T, E, k))
    moeq4.moe_route(logits, out, ws)
    return out


def _route_noalloc(logits, k, bm):
    T, E = logits.shape
    out = moeq4.RouteBuffers.alloc(T, E, k, bm)
    moeq4.moe_route_noalloc(logits, out)
    return out


def _same(a, b):
    torch.cuda.synchronize()
    for f in FIELDS:
        assert torch.equal(getattr(a, f), getattr(b, f)), f
    n = int(a.n_tiles[0])
    assert n == int(b.n_tiles[0])
    assert torch.equal(a.tiles[:n], b.tiles[:n])
    assert moeq4.moe_get_device_error(a) == 0 and moeq4.moe_get_device_error(b) == 0


def test_two_calls_match_workspace_routing():
    cfg = synth.CONFIGS["t4096"]
    for layer in (0, 1):   # two calls in a row on the shared scratch
        logits = torch.from_numpy(synth.gen_logits(cfg, layer)).cuda()
        _same(_route_noalloc(logits, cfg.k, 128), _route_ws(logits, cfg.k, 128))


def test_small_then_large_call():
    a = torch.from_numpy(np.random.default_rng(5).standard_normal((33, 40)).astype(np.float32)).cuda()
    _same(_route_noalloc(a, 5, 16), _route_ws(a, 5, 16))
    cfg = synth.CONFIGS["skew"]
    b = torch.from_numpy(synth.gen_logits(cfg)).cuda()
    _same(_route_noalloc(b, cfg.k, 128), _route_ws(b, cfg.k, 128))


def test_sizes_beyond_the_fixed_scratch_are_rejected():
    out = moeq4.RouteBuffers.alloc(8193, 16, 2, 128)
    logits = torch.zeros((8193, 16), dtype=torch.float32, device="cuda")
    with pytest.raises(moeq4.MoeError) as e:
        moeq4.moe_route_noalloc(logits, out)
    assert e.value.status == moeq4.MOE_ERR_TOO_LARGE


def test_limit_sizes_match_workspace_routing():
    # the largest sizes the fixed scratch is laid out for: T = 8192, E = 256, k = 8
    rng = np.random.default_rng(8192)
    a = torch.from_numpy(rng.standard_normal((8192, 256)).astype(np.float32)).cuda()
    for bm in (128, 64):
        _same(_route_noalloc(a, 8, bm), _route_ws(a, 8, bm))


@pytest.mark.parametrize("T,E,k", [(64, 257, 2), (64, 256, 9)])
def test_expert_and_topk_beyond_the_fixed_scratch_are_rejected(T, E, k):
    out = moeq4.RouteBuffers.alloc(T, E, k, 128)
    logits = torch.zeros((T, E), dtype=torch.float32, device="cuda")
    with pytest.raises(moeq4.MoeError) as e:
        moeq4.moe_route_noalloc(logits, out)
    assert e.value.status == moeq4.MOE_ERR_TOO_LARGE


def test_state_of_an_unfinished_call_is_ignored():
    # A call that did not finish (say, one that raced an overlapping call) can
    # leave count rows of its own in the fixed scratch. Plant such state, rows
    # full of wrong counts: the next call writes every row before reading it
    # and must route exactly as moe_route does.
    cfg = synth.CONFIGS["t512"]
    logits = torch.from_numpy(synth.gen_logits(cfg)).cuda()
    ref = _route_ws(logits, cfg.k, 128)
    _same(_route_noalloc(logits, cfg.k, 128), ref)
    addr, nbytes = moeq4.moe_debug_noalloc_scratch()

    class _Scratch:   # the library's array seen as an int32 tensor (no copy)
        __cuda_array_interface__ = {"shape": (nbytes // 4,), "typestr": "<i4",
                                    "data": (addr, False), "version": 3}

    scratch = torch.as_tensor(_Scratch(), device="cuda")
    torch.cuda.synchronize()
    scratch.fill_(777)                                    # count rows
    torch.cuda.synchronize()
    for _ in range(2):
        _same(_route_noalloc(logits, cfg.k, 128), ref)
