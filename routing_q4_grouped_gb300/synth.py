"""Seeded synthetic inputs for the prefill MoE expert layer.

This module only draws numbers: it holds none of the layer's arithmetic (no
dequantisation, routing or FFN math), so the CPU oracle and the CUDA path can
both be fed from it without sharing any computation.

Generator: a counter-based splitmix64 stream. For tensor ``tid`` of layer
``layer`` under seed ``seed`` the key is ``mix(mix(seed + G) ^ (tid << 32 | layer))``
and element ``i`` is ``mix(key + (i + 1) * G)`` with ``G = 0x9E3779B97F4A7C15``
and ``mix`` the splitmix64 finaliser (Steele, Lea and Flood, "Fast splittable
pseudorandom number generators", OOPSLA 2014). Uniforms take the top 53 bits;
normals use Box-Muller on two consecutive uniforms.

Workloads (the five layer configurations of the 4-bit MoE prefill study):

* ``tiny``    T=64,    d=256,  E=8,   k=2, f=128, no shared expert, seed 0
* ``t512``    T=512,   d=2048, E=256, k=8, f=512, shared f_s=512,   seed 1
* ``t4096``   T=4096,  same widths, per-expert logit offset 0.5*N(0,1), seed 2
* ``skew``    T=2048,  same widths, logits N(0,1) - 3*ln(rank_e),     seed 3
* ``chunked`` T=32768 in 4096-token chunks through 40 layers with independent
  weights and logits, seed 4

Value recipe shared by all: x ~ N(0,1) rounded to bf16; codes uniform on 0..15
packed 8 per uint32, low nibble first along K (uniform random 32-bit words are
exactly that); scale ~ U(0.004, 0.008) rounded to bf16; bias = -7.5*scale +
N(0, 0.001) rounded to bf16 (scale taken as its stored bf16 value).
"""
from __future__ import annotations

import dataclasses
import math

import numpy as np

_G = np.uint64(0x9E3779B97F4A7C15)
_M1 = np.uint64(0xBF58476D1CE4E5B9)
_M2 = np.uint64(0x94D049BB133111EB)

# Stable stream identifiers, one per generated tensor.
TID = {
    "x": 1, "logits": 2, "expert_bias": 3, "rank_perm": 4,
    "gu_qw": 10, "gu_scale": 11, "gu_bias": 12,
    "dn_qw": 13, "dn_scale": 14, "dn_bias": 15,
    "sgu_qw": 20, "sgu_scale": 21, "sgu_bias": 22,
    "sdn_qw": 23, "sdn_scale": 24, "sdn_bias": 25,
    "router": 30,
}


def _mix(z: np.ndarray) -> np.ndarray:
    z = (z ^ (z >> np.uint64(30))) * _M1
    z = (z ^ (z >> np.uint64(27))) * _M2
    return z ^ (z >> np.uint64(31))


def _key(seed: int, tid: int, layer: int) -> np.uint64:
    with np.errstate(over="ignore"):
        a = _mix(np.array([np.uint64(seed) + _G], dtype=np.uint64))[0]
        b = np.uint64((tid << 32) | (layer & 0xFFFFFFFF))
        return _mix(np.array([a ^ b], dtype=np.uint64))[0]


def u64_stream(seed: int, tid: int, layer: int, n: int, start: int = 0) -> np.ndarray:
    """Elements [start, start+n) of the counter-based stream."""
    key = _key(seed, tid, layer)
    i = np.arange(start + 1, start + n + 1, dtype=np.uint64)
    with np.errstate(over="ignore"):
        return _mix(key + i * _G)


def uniform(seed, tid, layer, n, start=0) -> np.ndarray:
    u = u64_stream(seed, tid, layer, n, start) >> np.uint64(11)
    return u.astype(np.float64) * (1.0 / 9007199254740992.0)


def normal(seed, tid, layer, n, start=0) -> np.ndarray:
    """Normals [start, start+n) of the stream (normal i uses uniforms 2i, 2i+1)."""
    u = uniform(seed, tid, layer, 2 * n, 2 * start)
    u1, u2 = u[0::2], u[1::2]
    return np.sqrt(-2.0 * np.log1p(-u1)) * np.cos(2.0 * math.pi * u2)


def to_bf16_bits(v: np.ndarray) -> np.ndarray:
    """Round to bf16 with PyTorch's converter and return the raw uint16 bits."""
    import torch

    t = torch.from_numpy(np.ascontiguousarray(v, dtype=np.float32)).to(torch.bfloat16)
    return t.view(torch.int16).numpy().view(np.uint16).copy()


def bf16_bits_to_f32(b: np.ndarray) -> np.ndarray:
    return (b.astype(np.uint32) << np.uint32(16)).view(np.float32)


@dataclasses.dataclass(frozen=True)
class Config:
    name: str
    T: int
    d: int
    E: int
    k: int
    f: int
    f_s: int
    seed: int
    logits: str = "normal"  # "normal" | "expert_offset" | "zipf"
    layers: int = 1
    chunk: int = 0  # tokens per chunk (0 = whole T at once)

    @property
    def tokens_per_call(self) -> int:
        return self.chunk if self.chunk else self.T


CONFIGS = {
    "tiny": Config("tiny", T=64, d=256, E=8, k=2, f=128, f_s=0, seed=0),
    "t512": Config("t512", T=512, d=2048, E=256, k=8, f=512, f_s=512, seed=1),
    "t4096": Config("t4096", T=4096, d=2048, E=256, k=8, f=512, f_s=512, seed=2,
                    logits="expert_offset"),
    "skew": Config("skew", T=2048, d=2048, E=256, k=8, f=512, f_s=512, seed=3, logits="zipf"),
    "chunked": Config("chunked", T=32768, d=2048, E=256, k=8, f=512, f_s=512, seed=4,
                      layers=40, chunk=4096),
}


def gen_x(cfg: Config, T: int | None = None, layer: int = 0, t0: int = 0) -> np.ndarray:
    """Token activations, bf16 bits [T, d] of tokens t0 .. t0+T-1 (``layer``
    selects an independent draw)."""
    T = cfg.T if T is None else T
    d = cfg.d
    return to_bf16_bits(normal(cfg.seed, TID["x"], layer, T * d, t0 * d).reshape(T, d))


def gen_logits(cfg: Config, layer: int = 0, T: int | None = None, t0: int = 0) -> np.ndarray:
    """Router logits, fp32 [T, E] of tokens t0 .. t0+T-1, following the
    configuration's recipe."""
    T = cfg.T if T is None else T
    E = cfg.E
    z = normal(cfg.seed, TID["logits"], layer, T * E, t0 * E).reshape(T, E)
    if cfg.logits == "expert_offset":
        z = z + 0.5 * normal(cfg.seed, TID["expert_bias"], layer, E)[None, :]
    elif cfg.logits == "zipf":
        perm = np.argsort(uniform(cfg.seed, TID["rank_perm"], layer, E), kind="stable")
        rank = np.empty(E, dtype=np.float64)
        rank[perm] = np.arange(1, E + 1, dtype=np.float64)
        z = z + 3.0 * (-np.log(rank))[None, :]
    return z.astype(np.float32)


def gen_router(cfg: Config, layer: int = 0) -> np.ndarray:
    """Router weights, bf16 bits [E, d] ~ N(0, 1/d): with x ~ N(0, 1) the logits
    x . Wr[e] are about N(0, 1), the spread the workloads' logits have."""
    d, E = cfg.d, cfg.E
    return to_bf16_bits(normal(cfg.seed, TID["router"], layer, E * d).reshape(E, d) / math.sqrt(d))


def _q4_matrix(seed, layer, prefix, experts, rows, K):
    """Packed codes [experts, rows, K/8] u32 and bf16 scale/bias [experts, rows, K/64]."""
    nwords = experts * rows * (K // 8)
    raw = u64_stream(seed, TID[prefix + "_qw"], layer, (nwords + 1) // 2)
    qw = raw.view(np.uint32)[:nwords].reshape(experts, rows, K // 8).copy()
    ng = experts * rows * (K // 64)
    s = 0.004 + 0.004 * uniform(seed, TID[prefix + "_scale"], layer, ng)
    s_bits = to_bf16_bits(s)
    s_val = bf16_bits_to_f32(s_bits).astype(np.float64)
    b = -7.5 * s_val + 0.001 * normal(seed, TID[prefix + "_bias"], layer, ng)
    b_bits = to_bf16_bits(b)
    shp = (experts, rows, K // 64)
    return qw, s_bits.reshape(shp), b_bits.reshape(shp)


@dataclasses.dataclass
class Q4Weights:
    """Packed weights of one layer (numpy, host).

    gate_up: [E, 2f, d/8] codes and [E, 2f, d/64] scale/bias; rows 0..f-1 are
    the gate projection and rows f..2f-1 the up projection.
    down:    [E, d, f/8] codes and [E, d, f/64] scale/bias.
    shared_*: the same for the always-on shared expert (E=1), or None.
    """
    E: int
    d: int
    f: int
    f_s: int
    gu_qw: np.ndarray
    gu_scale: np.ndarray
    gu_bias: np.ndarray
    dn_qw: np.ndarray
    dn_scale: np.ndarray
    dn_bias: np.ndarray
    sgu_qw: np.ndarray | None = None
    sgu_scale: np.ndarray | None = None
    sgu_bias: np.ndarray | None = None
    sdn_qw: np.ndarray | None = None
    sdn_scale: np.ndarray | None = None
    sdn_bias: np.ndarray | None = None

    @property
    def nbytes(self) -> int:
        tot = 0
        for f in dataclasses.fields(self):
            v = getattr(self, f.name)
            if isinstance(v, np.ndarray):
                tot += v.nbytes
        return tot


def gen_weights(cfg: Config, layer: int = 0) -> Q4Weights:
    E, d, f, fs, seed = cfg.E, cfg.d, cfg.f, cfg.f_s, cfg.seed
    gu = _q4_matrix(seed, layer, "gu", E, 2 * f, d)
    dn = _q4_matrix(seed, layer, "dn", E, d, f)
    kw = {}
    if fs:
        sgu = _q4_matrix(seed, layer, "sgu", 1, 2 * fs, d)
        sdn = _q4_matrix(seed, layer, "sdn", 1, d, fs)
        kw = dict(sgu_qw=sgu[0], sgu_scale=sgu[1], sgu_bias=sgu[2],
                  sdn_qw=sdn[0], sdn_scale=sdn[1], sdn_bias=sdn[2])
    return Q4Weights(E, d, f, fs, gu[0], gu[1], gu[2], dn[0], dn[1], dn[2], **kw)
