"""ctypes binding of libmoeq4 (C-ABI in include/moeq4.h), same names as the C calls.

Argument marshalling only: tensors are passed as raw device pointers, the
current CUDA stream as a handle, and every step of the layer runs in the
library's kernels. PyTorch provides device memory and streams. There is no
fallback: if the library is missing or the device is not sm_103 the calls
raise.
"""
from __future__ import annotations

import ctypes
import dataclasses
import os

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "_lib", "libmoeq4.so")

MOE_OK = 0
MOE_DEVERR_NONFINITE_LOGIT = 1
MOE_DEVERR_SCAN_TIMEOUT = 2
MOE_DEVERR_PIPE_TIMEOUT = 4
MOE_DEVERR_BAD_TILE = 8
MOE_DEVERR_BAD_WORKSPACE = 16
MOE_ERR_TOO_LARGE = -8

_c_i32 = ctypes.c_int32
_c_ptr = ctypes.c_void_p
_c_size = ctypes.c_size_t


class Q4Mat(ctypes.Structure):
    _fields_ = [("qw", _c_ptr), ("scale", _c_ptr), ("bias", _c_ptr)]


class Q4WeightsC(ctypes.Structure):
    _fields_ = [("gate_up", Q4Mat), ("down", Q4Mat), ("sh_gate_up", Q4Mat), ("sh_down", Q4Mat),
                ("E", _c_i32), ("d", _c_i32), ("f", _c_i32), ("f_s", _c_i32)]


class Q4PackedC(ctypes.Structure):
    _fields_ = [("data", _c_ptr), ("E", _c_i32), ("d", _c_i32), ("f", _c_i32), ("f_s", _c_i32)]


class RouteOutC(ctypes.Structure):
    _fields_ = [("ids", _c_ptr), ("w", _c_ptr), ("counts", _c_ptr), ("offsets", _c_ptr),
                ("perm", _c_ptr), ("inv", _c_ptr), ("tiles", _c_ptr), ("n_tiles", _c_ptr),
                ("err", _c_ptr), ("T", _c_i32), ("E", _c_i32), ("k", _c_i32),
                ("block_m", _c_i32)]


class MoeError(RuntimeError):
    def __init__(self, fn, status):
        self.status = status
        super().__init__(f"{fn}: {status_string(status)} ({status})")


_lib = None

_SIGS = {
    "moe_route_max_tiles": (_c_i32, [_c_i32, _c_i32, _c_i32, _c_i32]),
    "moe_route_workspace_size": (_c_size, [_c_i32, _c_i32, _c_i32]),
    "moe_ffn_workspace_size": (_c_size, [_c_i32] * 7),
    "moe_layer_workspace_size": (_c_size, [_c_i32] * 7),
    "moe_route": (_c_i32, [_c_ptr, ctypes.POINTER(RouteOutC), _c_ptr, _c_size, _c_ptr]),
    "moe_route_noalloc": (_c_i32, [_c_ptr, ctypes.POINTER(RouteOutC), _c_ptr]),
    "moe_q4_packed_size": (_c_size, [_c_i32] * 4),
    "moe_q4_prepack": (_c_i32, [ctypes.POINTER(Q4WeightsC), _c_ptr, _c_size, _c_ptr]),
    "moe_expert_ffn": (_c_i32, [_c_ptr, _c_i32, _c_i32, ctypes.POINTER(Q4PackedC),
                                ctypes.POINTER(RouteOutC), _c_ptr, _c_ptr, _c_size, _c_ptr]),
    "moe_layer": (_c_i32, [_c_ptr, _c_ptr, _c_i32, ctypes.POINTER(Q4PackedC),
                           ctypes.POINTER(RouteOutC), _c_ptr, _c_ptr, _c_size, _c_ptr]),
    "moe_expert_ffn_decode": (_c_i32, [_c_ptr, _c_i32, _c_i32, ctypes.POINTER(Q4PackedC),
                                       ctypes.POINTER(RouteOutC), _c_ptr, _c_ptr, _c_size, _c_ptr]),
    "moe_debug_set_decode_max_t": (_c_i32, [_c_i32]),
    "moe_router_topk": (_c_i32, [_c_ptr, _c_ptr, _c_i32, _c_i32, _c_ptr,
                                 ctypes.POINTER(RouteOutC), _c_ptr]),
    "moe_route_ids": (_c_i32, [ctypes.POINTER(RouteOutC), _c_ptr, _c_size, _c_ptr]),
    "moe_layer_router": (_c_i32, [_c_ptr, _c_ptr, _c_i32, ctypes.POINTER(Q4PackedC), _c_ptr,
                                  ctypes.POINTER(RouteOutC), _c_ptr, _c_ptr, _c_size, _c_ptr]),
    "moe_l2_prefetch": (_c_i32, [_c_ptr, _c_size, _c_ptr]),

    "moe_get_device_error": (_c_i32, [_c_ptr, ctypes.POINTER(_c_i32), _c_ptr]),
    "moe_status_string": (ctypes.c_char_p, [_c_i32]),
    "moe_residual_rms": (_c_i32, [_c_ptr, _c_ptr, _c_ptr, _c_i32, _c_i32, _c_ptr]),
    "moe_debug_dequant": (_c_i32, [_c_ptr, _c_ptr, _c_ptr, _c_i32, _c_i32, _c_ptr, _c_ptr]),
    "moe_debug_mma": (_c_i32, [_c_i32, _c_ptr, _c_ptr, _c_ptr, _c_i32, _c_i32, _c_ptr]),
    "moe_debug_set_stage_events": (_c_i32, [ctypes.POINTER(_c_ptr), _c_i32]),
    "moe_debug_tmem_layout": (_c_i32, [_c_ptr, _c_ptr]),
    "moe_debug_noalloc_scratch": (_c_i32, [ctypes.POINTER(_c_ptr), ctypes.POINTER(_c_size)]),
}


def lib() -> ctypes.CDLL:
    """Loads libmoeq4.so (built in-tree); raises if it has not been built."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(f"{LIB_PATH} is missing: run `python -m routing_q4_grouped_gb300.build`")
        L = ctypes.CDLL(LIB_PATH)
        for name, (res, args) in _SIGS.items():
            fn = getattr(L, name)
            fn.restype = res
            fn.argtypes = args
        _lib = L
    return _lib


def status_string(s: int) -> str:
    return lib().moe_status_string(s).decode()


def _check(fn, s):
    if s != MOE_OK:
        raise MoeError(fn, s)


def _ptr(t) -> int | None:
    return None if t is None else t.data_ptr()


def _need(fn, t, dtype, name, optional=False):
    """The library reads every array as a dense row-major device buffer."""
    if t is None and optional:
        return
    if t is None or not t.is_cuda or t.dtype != dtype or not t.is_contiguous():
        got = "None" if t is None else f"{t.dtype} on {t.device}, contiguous={t.is_contiguous()}"
        raise ValueError(f"{fn}: {name} must be a contiguous {dtype} CUDA tensor, got {got}")


def _stream(stream) -> int:
    s = torch.cuda.current_stream() if stream is None else stream
    return s.cuda_stream


# ----------------------------------------------------------------- host-side sizes

def moe_route_max_tiles(T, E, k, block_m) -> int:
    return lib().moe_route_max_tiles(T, E, k, block_m)


def moe_route_workspace_size(T, E, k) -> int:
    return lib().moe_route_workspace_size(T, E, k)


def moe_ffn_workspace_size(T, E, k, d, f, f_s, block_m=128) -> int:
    return lib().moe_ffn_workspace_size(T, E, k, d, f, f_s, block_m)


def moe_layer_workspace_size(T, E, k, d, f, f_s, block_m=128) -> int:
    return lib().moe_layer_workspace_size(T, E, k, d, f, f_s, block_m)


# ------------------------------------------------------------------ device buffers

def moe_q4_packed_size(E, d, f, f_s) -> int:
    return lib().moe_q4_packed_size(E, d, f, f_s)


def moe_q4_prepack(W: "DeviceWeights", dst: torch.Tensor, stream=None) -> None:
    """Reorders the interchange-layout device weights of W into dst (kernel-native)."""
    wc = W.interchange_cstruct()
    _check("moe_q4_prepack", lib().moe_q4_prepack(ctypes.byref(wc), _ptr(dst), dst.numel(),
                                                  _stream(stream)))


@dataclasses.dataclass
class DeviceWeights:
    """One layer's 4-bit weights on the GPU: the kernel-native copy the layer
    streams (``packed``) and, until :meth:`drop_interchange`, the interchange
    arrays it was made from (torch tensors as storage)."""
    E: int
    d: int
    f: int
    f_s: int
    tensors: dict
    packed: torch.Tensor = None

    @classmethod
    def from_host(cls, W, device="cuda", keep_interchange=False):
        """Copies a :class:`routing_q4_grouped_gb300.synth.Q4Weights` to the device and prepacks it."""
        names = ["gu_qw", "gu_scale", "gu_bias", "dn_qw", "dn_scale", "dn_bias"]
        if W.f_s:
            names += ["sgu_qw", "sgu_scale", "sgu_bias", "sdn_qw", "sdn_scale", "sdn_bias"]
        ts = {}
        for n in names:
            a = getattr(W, n)
            t = torch.from_numpy(a.view(a.dtype.str.replace("u", "i")) if a.dtype.kind == "u" else a)
            ts[n] = t.to(device)
        dw = cls(W.E, W.d, W.f, W.f_s, ts)
        dw.packed = torch.empty(moe_q4_packed_size(W.E, W.d, W.f, W.f_s), dtype=torch.uint8,
                                device=device)
        moe_q4_prepack(dw, dw.packed)
        if not keep_interchange:
            torch.cuda.current_stream().synchronize()
            dw.tensors = {}
        return dw

    def interchange_cstruct(self) -> Q4WeightsC:
        t = self.tensors
        if not t:
            raise RuntimeError("interchange arrays were dropped after prepacking")
        m = lambda p: Q4Mat(_ptr(t.get(p + "_qw")), _ptr(t.get(p + "_scale")), _ptr(t.get(p + "_bias")))
        return Q4WeightsC(m("gu"), m("dn"), m("sgu") if self.f_s else Q4Mat(),
                          m("sdn") if self.f_s else Q4Mat(), self.E, self.d, self.f, self.f_s)

    def cstruct(self) -> Q4PackedC:
        return Q4PackedC(_ptr(self.packed), self.E, self.d, self.f, self.f_s)

    @property
    def nbytes(self) -> int:
        return self.packed.numel()


@dataclasses.dataclass
class RouteBuffers:
    """Device arrays of a routing result (see moe_route_out in moeq4.h)."""
    T: int
    E: int
    k: int
    block_m: int
    ids: torch.Tensor
    w: torch.Tensor
    counts: torch.Tensor
    offsets: torch.Tensor
    perm: torch.Tensor
    inv: torch.Tensor
    tiles: torch.Tensor
    n_tiles: torch.Tensor
    err: torch.Tensor

    @classmethod
    def alloc(cls, T, E, k, block_m=128, device="cuda"):
        i32 = dict(dtype=torch.int32, device=device)
        nmax = max(1, moe_route_max_tiles(T, E, k, block_m))
        return cls(T, E, k, block_m,
                   ids=torch.empty((T, k), **i32),
                   w=torch.empty((T, k), dtype=torch.float32, device=device),
                   counts=torch.empty(E, **i32), offsets=torch.empty(E + 1, **i32),
                   perm=torch.empty(max(1, T * k), **i32), inv=torch.empty(max(1, T * k), **i32),
                   tiles=torch.empty((nmax, 3), **i32), n_tiles=torch.zeros(4, **i32),
                   err=torch.zeros(4, **i32))

    def cstruct(self) -> RouteOutC:
        return RouteOutC(_ptr(self.ids), _ptr(self.w), _ptr(self.counts), _ptr(self.offsets),
                         _ptr(self.perm), _ptr(self.inv), _ptr(self.tiles), _ptr(self.n_tiles),
                         _ptr(self.err), self.T, self.E, self.k, self.block_m)


def alloc_workspace(nbytes: int, device="cuda") -> torch.Tensor:
    """Zero-filled scratch (the FFN part's grid-barrier counter must start at zero)."""
    return torch.zeros(max(nbytes, 256), dtype=torch.uint8, device=device)


# ---------------------------------------------------------------------- compute

def moe_route(logits: torch.Tensor, out: RouteBuffers, ws: torch.Tensor, stream=None) -> None:
    """Routing of fp32 logits [T, E] into ``out`` (asynchronous)."""
    _need("moe_route", logits, torch.float32, "logits")
    c = out.cstruct()
    _check("moe_route", lib().moe_route(_ptr(logits), ctypes.byref(c), _ptr(ws), ws.numel(),
                                        _stream(stream)))


def moe_route_noalloc(logits: torch.Tensor, out: RouteBuffers, stream=None) -> None:
    """moe_route with the library's fixed internal scratch (no workspace argument).

    For callers that cannot allocate device memory; limited to T <= 8192,
    E <= 256, k <= 8. Calls that overlap on the GPU share the scratch and race.
    """
    _need("moe_route_noalloc", logits, torch.float32, "logits")
    c = out.cstruct()
    _check("moe_route_noalloc", lib().moe_route_noalloc(_ptr(logits), ctypes.byref(c), _stream(stream)))


def moe_expert_ffn(x: torch.Tensor, W: DeviceWeights, r: RouteBuffers, y: torch.Tensor,
                   ws: torch.Tensor, stream=None) -> None:
    """Grouped expert FFN: bf16 x [T, d] -> bf16 y [T, d] (asynchronous)."""
    _need("moe_expert_ffn", x, torch.bfloat16, "x")
    _need("moe_expert_ffn", y, torch.bfloat16, "y")
    T, d = x.shape
    wc, rc = W.cstruct(), r.cstruct()
    _check("moe_expert_ffn", lib().moe_expert_ffn(_ptr(x), T, d, ctypes.byref(wc), ctypes.byref(rc),
                                                  _ptr(y), _ptr(ws), ws.numel(), _stream(stream)))


def moe_expert_ffn_decode(x: torch.Tensor, W: DeviceWeights, r: RouteBuffers, y: torch.Tensor,
                          ws: torch.Tensor, stream=None) -> None:
    """The small-batch expert FFN (T <= 64): split-K weight streaming on the CUDA cores."""
    _need("moe_expert_ffn_decode", x, torch.bfloat16, "x")
    _need("moe_expert_ffn_decode", y, torch.bfloat16, "y")
    T, d = x.shape
    wc, rc = W.cstruct(), r.cstruct()
    _check("moe_expert_ffn_decode",
           lib().moe_expert_ffn_decode(_ptr(x), T, d, ctypes.byref(wc), ctypes.byref(rc), _ptr(y),
                                       _ptr(ws), ws.numel(), _stream(stream)))


def moe_debug_set_decode_max_t(t: int) -> None:
    """Batches of at most t tokens take the decode path in moe_expert_ffn / moe_layer (0 = never)."""
    _check("moe_debug_set_decode_max_t", lib().moe_debug_set_decode_max_t(t))


def moe_layer(x: torch.Tensor, logits: torch.Tensor, W: DeviceWeights, r: RouteBuffers,
              y: torch.Tensor, ws: torch.Tensor, stream=None) -> None:
    """Routing then expert FFN on one stream, no host synchronisation."""
    _need("moe_layer", x, torch.bfloat16, "x")
    _need("moe_layer", logits, torch.float32, "logits")
    _need("moe_layer", y, torch.bfloat16, "y")
    T = x.shape[0]
    wc, rc = W.cstruct(), r.cstruct()
    _check("moe_layer", lib().moe_layer(_ptr(x), _ptr(logits), T, ctypes.byref(wc), ctypes.byref(rc),
                                        _ptr(y), _ptr(ws), ws.numel(), _stream(stream)))


def moe_router_topk(x: torch.Tensor, w_router: torch.Tensor, out: RouteBuffers,
                    logits: torch.Tensor = None, stream=None) -> None:
    """Router projection x [T, d] . w_router [E, d]^T with the top-k fused:
    writes out.ids / out.w (and logits [T, E] fp32 when given)."""
    _need("moe_router_topk", x, torch.bfloat16, "x")
    _need("moe_router_topk", w_router, torch.bfloat16, "w_router")
    _need("moe_router_topk", logits, torch.float32, "logits", optional=True)
    T, d = x.shape
    rc = out.cstruct()
    _check("moe_router_topk", lib().moe_router_topk(_ptr(x), _ptr(w_router), T, d, _ptr(logits),
                                                    ctypes.byref(rc), _stream(stream)))


def moe_route_ids(out: RouteBuffers, ws: torch.Tensor, stream=None) -> None:
    """Histogram, scan, scatter and block map from out.ids / out.w."""
    rc = out.cstruct()
    _check("moe_route_ids", lib().moe_route_ids(ctypes.byref(rc), _ptr(ws), ws.numel(),
                                                _stream(stream)))


def moe_layer_router(x: torch.Tensor, w_router: torch.Tensor, W: DeviceWeights, r: RouteBuffers,
                     y: torch.Tensor, ws: torch.Tensor, logits: torch.Tensor = None,
                     stream=None) -> None:
    """The layer from hidden states: fused router, routing from its choice, expert FFN."""
    _need("moe_layer_router", x, torch.bfloat16, "x")
    _need("moe_layer_router", w_router, torch.bfloat16, "w_router")
    _need("moe_layer_router", y, torch.bfloat16, "y")
    _need("moe_layer_router", logits, torch.float32, "logits", optional=True)
    T = x.shape[0]
    wc, rc = W.cstruct(), r.cstruct()
    _check("moe_layer_router", lib().moe_layer_router(_ptr(x), _ptr(w_router), T, ctypes.byref(wc),
                                                      _ptr(logits), ctypes.byref(rc), _ptr(y),
                                                      _ptr(ws), ws.numel(), _stream(stream)))


def moe_residual_rms(y: torch.Tensor, x: torch.Tensor, out: torch.Tensor, stream=None) -> None:
    """Next layer's input of the chunked run: bf16((y + x) / rms(y + x)) per token."""
    for name, t in (("y", y), ("x", x), ("out", out)):
        _need("moe_residual_rms", t, torch.bfloat16, name)
    T, d = x.shape
    _check("moe_residual_rms", lib().moe_residual_rms(_ptr(y), _ptr(x), _ptr(out), T, d,
                                                      _stream(stream)))


def moe_l2_prefetch(t: torch.Tensor, nbytes: int = None, stream=None) -> None:
    """Prefetch the first nbytes (default all) of device tensor t into L2."""
    n = t.numel() * t.element_size() if nbytes is None else min(nbytes, t.numel() * t.element_size())
    n -= n % 16
    _check("moe_l2_prefetch", lib().moe_l2_prefetch(_ptr(t), n, _stream(stream)))


def moe_get_device_error(r: RouteBuffers, stream=None) -> int:
    """Synchronises the stream and returns the device error word (0 = none)."""
    code = _c_i32(0)
    s = lib().moe_get_device_error(_ptr(r.err), ctypes.byref(code), _stream(stream))
    if s not in (MOE_OK, -5):
        raise MoeError("moe_get_device_error", s)
    return code.value


# ----------------------------------------------------------------- test-only calls

def moe_debug_dequant(qw, scale, bias, out, stream=None) -> None:
    rows, K = out.shape
    _check("moe_debug_dequant", lib().moe_debug_dequant(_ptr(qw), _ptr(scale), _ptr(bias), rows, K,
                                                        _ptr(out), _stream(stream)))


def moe_debug_mma(a_from_tmem: bool, A, B, D, stream=None) -> None:
    N, K = B.shape
    _check("moe_debug_mma", lib().moe_debug_mma(int(a_from_tmem), _ptr(A), _ptr(B), _ptr(D), N, K,
                                                _stream(stream)))


def moe_debug_tmem_layout(out, stream=None) -> None:
    _check("moe_debug_tmem_layout", lib().moe_debug_tmem_layout(_ptr(out), _stream(stream)))


def moe_debug_noalloc_scratch() -> tuple[int, int]:
    """(device address, bytes) of moe_route_noalloc's fixed scratch on the current device."""
    addr, n = _c_ptr(), _c_size()
    _check("moe_debug_noalloc_scratch",
           lib().moe_debug_noalloc_scratch(ctypes.byref(addr), ctypes.byref(n)))
    return int(addr.value), int(n.value)


def moe_debug_set_stage_events(events) -> None:
    """Registers torch.cuda.Event objects recorded at the layer's stage boundaries."""
    arr = (_c_ptr * max(1, len(events)))(*[e.cuda_event for e in events])
    _check("moe_debug_set_stage_events", lib().moe_debug_set_stage_events(arr, len(events)))


def default_block_m(T: int, E: int, k: int) -> int:
    """Tile height of the block map for a batch of T tokens: 64 when the expert
    groups average at most 32 rows (short groups, weights streamed from HBM:
    the 64-row kernels keep a deeper tensor-memory pipeline), else 128 (every
    weight tile expanded once per 128 token rows)."""
    return 64 if T * k <= 32 * E else 128


class Layer:
    """Convenience owner of the buffers one layer call needs (T tokens);
    block_m=None picks default_block_m(T, E, k)."""

    def __init__(self, W: DeviceWeights, T: int, k: int, block_m=128, device="cuda"):
        if block_m is None:
            block_m = default_block_m(T, W.E, k)
        self.W, self.T, self.k = W, T, k
        self.route = RouteBuffers.alloc(T, W.E, k, block_m, device)
        self.ws = alloc_workspace(moe_layer_workspace_size(T, W.E, k, W.d, W.f, W.f_s, block_m), device)
        self.y = torch.empty((T, W.d), dtype=torch.bfloat16, device=device)

    def __call__(self, x, logits, stream=None):
        moe_layer(x, logits, self.W, self.route, self.y, self.ws, stream)
        return self.y
