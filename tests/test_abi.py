"""The C-ABI library loads on a machine without a GPU, exports every symbol the
headers declare, and rejects bad arguments on the host before touching a device."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADERS = [os.path.join(ROOT, "include", h) for h in ("moeq4.h", "moeq4_debug.h")]


@pytest.fixture(scope="module")
def L():
    from routing_q4_grouped_gb300 import build, moeq4
    if not os.path.exists(moeq4.LIB_PATH):
        build.build()
    return moeq4


def _declared():
    names = set()
    for h in HEADERS:
        src = open(h).read()
        src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
        for m in re.finditer(r"^\s*[a-zA-Z_][\w \*]*?\b(moe_\w+)\s*\(", src, flags=re.M):
            names.add(m.group(1))
    return names


def test_headers_declare_the_boundary():
    names = _declared()
    for n in ("moe_route", "moe_expert_ffn", "moe_layer", "moe_route_max_tiles",
              "moe_route_workspace_size", "moe_ffn_workspace_size", "moe_layer_workspace_size",
              "moe_get_device_error", "moe_status_string", "moe_residual_rms",
              "moe_q4_packed_size", "moe_q4_prepack", "moe_debug_dequant", "moe_debug_mma",
              "moe_debug_set_stage_events", "moe_debug_tmem_layout"):
        assert n in names, n


def test_library_exports_every_declared_symbol(L):
    lib = ctypes.CDLL(L.LIB_PATH)
    missing = [n for n in sorted(_declared()) if not hasattr(lib, n)]
    assert not missing, missing


def test_host_side_sizes(L):
    assert L.moe_route_max_tiles(4096, 256, 8, 128) == 4096 * 8 // 128 + 256
    assert L.moe_route_max_tiles(3, 4, 2, 2) == 3 + 4
    assert L.moe_route_workspace_size(4096, 256, 8) > 4096 * 8 * 4
    ffn = L.moe_ffn_workspace_size(4096, 256, 8, 2048, 512, 512, 128)
    assert ffn >= 4096 * 8 * 512 * 2 + 4096 * 512 * 2 + 4096 * 2048 * 4
    lay = L.moe_layer_workspace_size(4096, 256, 8, 2048, 512, 512, 128)
    assert lay >= ffn + L.moe_route_workspace_size(4096, 256, 8)
    assert L.status_string(0) == "ok"
    assert "workspace" in L.status_string(-3)


def test_route_workspace_is_one_count_row_per_block(L):
    # the routing scratch holds one row of per-expert counts (uint32, rows padded
    # to 4 experts for 16-byte loads) per block of at least 8 tokens, and nothing
    # else: there are no counters to zero between calls
    def expect(T, E):
        blocks = max(1, -(-T // 8))
        rows = blocks * (-(-E // 4) * 4) * 4
        return -(-rows // 256) * 256
    for T, E in [(0, 256), (1, 256), (8, 256), (9, 256), (4096, 256), (100000, 256),
                 (300, 1000), (5, 17)]:
        assert L.moe_route_workspace_size(T, E, 8) == expect(T, E), (T, E)


def test_router_and_prefetch_arguments_rejected_on_host(L):
    lib = L.lib()
    fake = 1 << 20
    assert lib.moe_l2_prefetch(None, 16, None) == -1                  # no pointer
    assert lib.moe_l2_prefetch(fake + 8, 16, None) == -7              # misaligned start
    assert lib.moe_l2_prefetch(fake, 24, None) == -7                  # length not a multiple of 16
    assert lib.moe_l2_prefetch(fake, 0, None) == 0                    # nothing to do
    r = L.RouteOutC()
    for f in ("ids", "w", "counts", "offsets", "perm", "inv", "tiles", "n_tiles", "err"):
        setattr(r, f, fake)
    r.T, r.E, r.k, r.block_m = 16, 256, 9, 128                        # k above the router's 8
    assert lib.moe_router_topk(fake, fake, 16, 2048, fake, ctypes.byref(r), None) == -2
    r.E, r.k = 250, 8                                                 # E not a multiple of 16
    assert lib.moe_router_topk(fake, fake, 16, 2048, fake, ctypes.byref(r), None) == -2
    r.E = 256
    assert lib.moe_router_topk(fake, fake, 16, 2000, fake, ctypes.byref(r), None) == -2   # d % 64
    assert lib.moe_router_topk(fake, fake, 15, 2048, fake, ctypes.byref(r), None) == -2   # T mismatch
    assert lib.moe_router_topk(None, fake, 16, 2048, fake, ctypes.byref(r), None) == -1   # no x
    assert lib.moe_router_topk(fake, fake, 16, 2048, fake + 4, ctypes.byref(r), None) == -7
    assert lib.moe_route_ids(ctypes.byref(r), fake, 0, None) == -3   # workspace too small
    assert lib.moe_debug_set_decode_max_t(-1) == -1


def test_bad_arguments_rejected_on_host(L):
    lib = L.lib()
    r = L.RouteOutC()                       # all NULL
    r.T, r.E, r.k, r.block_m = 16, 8, 2, 128
    assert lib.moe_route(None, ctypes.byref(r), None, 0, None) == -1      # MOE_ERR_ARG
    fake = 1 << 20                          # aligned non-null values, never dereferenced
    for f in ("ids", "w", "counts", "offsets", "perm", "inv", "tiles", "n_tiles", "err"):
        setattr(r, f, fake)
    r.k = 9                                 # k > E
    assert lib.moe_route(fake, ctypes.byref(r), fake, 1 << 30, None) == -1
    r.k, r.block_m = 2, 129                 # block_m above the supported maximum
    assert lib.moe_route(fake, ctypes.byref(r), fake, 1 << 30, None) == -1
    r.block_m = 128
    assert lib.moe_route(fake, ctypes.byref(r), fake, 0, None) == -3      # workspace too small
    assert lib.moe_route(fake + 4, ctypes.byref(r), fake, 1 << 30, None) == -7   # misaligned
    P = L.Q4PackedC(fake, 8, 200, 128, 0)   # d not a multiple of 256
    assert lib.moe_expert_ffn(fake, 16, 200, ctypes.byref(P), ctypes.byref(r), fake, fake,
                              1 << 30, None) == -2
    P = L.Q4PackedC(None, 8, 256, 128, 0)   # no weight buffer
    assert lib.moe_expert_ffn(fake, 16, 256, ctypes.byref(P), ctypes.byref(r), fake, fake,
                              1 << 30, None) == -1
    W = L.Q4WeightsC()
    W.E, W.d, W.f, W.f_s = 8, 256, 128, 128  # shared expert declared but pointers NULL
    for m in (W.gate_up, W.down):
        m.qw = m.scale = m.bias = fake
    assert lib.moe_q4_prepack(ctypes.byref(W), fake, 1 << 30, None) == -1
    W.f_s = 0
    assert lib.moe_q4_prepack(ctypes.byref(W), fake, 16, None) == -3   # destination too small
    # the kernel-native copy has exactly the bytes of the interchange arrays
    E, d, f, fs = 256, 2048, 512, 512
    inter = (E * 2 * f * d // 2 + E * 2 * f * (d // 64) * 4 + E * d * f // 2 + E * d * (f // 64) * 4
             + 2 * fs * d // 2 + 2 * fs * (d // 64) * 4 + d * fs // 2 + d * (fs // 64) * 4)
    assert L.moe_q4_packed_size(E, d, f, fs) == inter


def test_ffn_and_layer_arguments_rejected_on_host(L):
    lib = L.lib()
    fake = 1 << 20                          # aligned non-null values, never dereferenced
    r = L.RouteOutC()
    for f in ("ids", "w", "counts", "offsets", "perm", "inv", "tiles", "n_tiles", "err"):
        setattr(r, f, fake)
    r.T, r.E, r.k, r.block_m = 16, 8, 2, 128
    P = L.Q4PackedC(fake, 8, 256, 128, 0)
    big = 1 << 30
    ffn = lambda x, T, d, y, ws, n: lib.moe_expert_ffn(x, T, d, ctypes.byref(P), ctypes.byref(r),
                                                      y, ws, n, None)
    assert ffn(None, 16, 256, fake, fake, big) == -1          # x NULL with T > 0
    assert ffn(fake, 16, 256, None, fake, big) == -1          # y NULL with T > 0
    assert ffn(fake, 16, 256, fake, None, big) == -1          # no workspace
    assert ffn(fake + 8, 16, 256, fake, fake, big) == -7      # x not 16-byte aligned
    assert ffn(fake, 15, 256, fake, fake, big) == -2          # T differs from the routing result
    assert ffn(fake, 16, 512, fake, fake, big) == -2          # d differs from the weights
    assert ffn(fake, 16, 256, fake, fake, 64) == -3           # workspace too small
    r.E = 16                                                  # routing over more experts than W has
    assert ffn(fake, 16, 256, fake, fake, big) == -2
    r.E = 8
    lay = lambda x, lg, T, y, ws, n: lib.moe_layer(x, lg, T, ctypes.byref(P), ctypes.byref(r),
                                                   y, ws, n, None)
    assert lay(fake, fake, 15, fake, fake, big) == -2         # T differs from r.T
    assert lay(fake, fake, 16, fake, None, big) == -3         # no workspace
    assert lay(fake, fake, 16, fake, fake, 64) == -3          # workspace too small
    assert lay(None, fake, 16, fake, fake, big) == -1         # x NULL with T > 0
    assert lay(fake, fake, 16, None, fake, big) == -1         # y NULL with T > 0
    # the FFN's alignment rules are checked before the routing is enqueued
    assert lay(fake + 8, fake, 16, fake, fake, big) == -7     # x not 16-byte aligned
    assert lay(fake, fake, 16, fake + 8, fake, big) == -7     # y not 16-byte aligned
    r.E = 16
    assert lay(fake, fake, 16, fake, fake, big) == -2         # expert counts differ
    # the layer from hidden states checks everything before the router is enqueued
    P16 = L.Q4PackedC(fake, 16, 256, 128, 0)
    lr = lambda x, y, ws: lib.moe_layer_router(x, fake, 16, ctypes.byref(P16), fake,
                                               ctypes.byref(r), y, ws, big, None)
    assert lr(fake, fake, fake + 8) == -7                     # workspace not 16-byte aligned
    assert lr(fake, fake + 8, fake) == -7                     # y not 16-byte aligned
    assert lr(None, fake, fake) == -1                         # x NULL with T > 0


def test_binding_rejects_host_or_strided_tensors_before_the_library():
    # the binding hands raw pointers to the library, which reads dense row-major
    # device arrays: anything else is refused in Python, before any call
    import torch
    from routing_q4_grouped_gb300 import moeq4
    x = torch.zeros((4, 256), dtype=torch.bfloat16)
    lg = torch.zeros((4, 8), dtype=torch.float32)
    with pytest.raises(ValueError, match="moe_layer: x must be a contiguous torch.bfloat16 CUDA"):
        moeq4.moe_layer(x, lg, None, None, x, None)
    with pytest.raises(ValueError, match="moe_route: logits must be .* torch.float32"):
        moeq4.moe_route(lg.double(), None, None)
    with pytest.raises(ValueError, match="moe_router_topk: x must be"):
        moeq4.moe_router_topk(x, None, None)
    with pytest.raises(ValueError, match="moe_residual_rms: y must be"):
        moeq4.moe_residual_rms(x, x.t(), x)
    assert not moeq4._need("f", None, torch.float32, "logits", optional=True)
    with pytest.raises(ValueError, match="got None"):
        moeq4._need("f", None, torch.float32, "logits")
