"""Shared helpers of the GPU parity tests (host <-> device marshalling, tolerances)."""
import numpy as np
import torch

import oracle as O
from routing_q4_grouped_gb300 import moeq4, synth

# Tolerance of the layer output against the oracle (fixed by the layer specification).
REL_L2_MAX = 5e-3
MAX_ABS_FRAC = 3e-2


def dev(a: np.ndarray) -> torch.Tensor:
    if a.dtype == np.uint16:
        return torch.from_numpy(a.view(np.int16)).cuda().view(torch.bfloat16)
    if a.dtype == np.uint32:
        return torch.from_numpy(a.view(np.int32)).cuda()
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


def bits(t: torch.Tensor) -> np.ndarray:
    return t.contiguous().view(torch.int16).cpu().numpy().view(np.uint16)


def route_gpu(logits: np.ndarray, k: int, block_m: int, ws=None):
    T, E = logits.shape
    out = moeq4.RouteBuffers.alloc(T, E, k, block_m)
    if ws is None:
        ws = moeq4.alloc_workspace(moeq4.moe_route_workspace_size(T, E, k))
    moeq4.moe_route(dev(logits) if T else torch.empty((0, E), device="cuda"), out, ws)
    err = moeq4.moe_get_device_error(out)
    return out, err, ws


def route_np(out):
    n = int(out.n_tiles[0].item())
    return dict(ids=out.ids.cpu().numpy(), w=out.w.cpu().numpy(), counts=out.counts.cpu().numpy(),
                offsets=out.offsets.cpu().numpy(), perm=out.perm.cpu().numpy()[: out.T * out.k],
                inv=out.inv.cpu().numpy()[: out.T * out.k], tiles=out.tiles.cpu().numpy()[:n],
                n_tiles=n)


def ulp_diff_f32(a: np.ndarray, b: np.ndarray) -> np.ndarray:
    ia = a.astype(np.float32).view(np.int32).astype(np.int64)
    ib = b.astype(np.float32).view(np.int32).astype(np.int64)
    return np.abs(ia - ib)


def assert_route_equal(g: dict, r: O.Route):
    assert np.array_equal(g["ids"], r.ids)
    assert np.array_equal(g["counts"], r.counts)
    assert np.array_equal(g["offsets"], r.offsets)
    assert np.array_equal(g["perm"], r.perm)
    assert np.array_equal(g["inv"], r.inv)
    assert g["n_tiles"] == r.n_tiles
    assert np.array_equal(g["tiles"], r.tiles)
    # weights: float64 on both sides, then one rounding to fp32: bit-exact
    assert np.array_equal(g["w"].view(np.uint32), r.w.view(np.uint32)), \
        ulp_diff_f32(g["w"], r.w).max(initial=0)


def assert_y_close(y_gpu: np.ndarray, y_ref: np.ndarray):
    g = O.bf16_value(y_gpu)
    r = O.bf16_value(y_ref)
    assert np.all(np.isfinite(g))
    rel = np.linalg.norm(g - r) / max(np.linalg.norm(r), 1e-30)
    mx = np.abs(g - r).max(initial=0.0)
    assert rel <= REL_L2_MAX, rel
    assert mx <= MAX_ABS_FRAC * np.abs(r).max(initial=0.0), (mx, np.abs(r).max())
    return rel, mx
