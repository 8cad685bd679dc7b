"""CPU oracle for the prefill MoE expert layer (4-bit grouped weights, GPU-style routing).

TEST INFRASTRUCTURE ONLY. This package is the plain, slow, obviously correct
restatement of what the layer computes. Only the test suite, the smoke check
and the benchmark's CPU-baseline / reference legs may import it; the product
path (the CUDA library and its binding) never does, and it shares no code,
table or helper with that path.

Sources (web pages on Perplexity's "Lily" engine; cited by title and section):

* [A] "Perplexity Lily 오픈소스 공개 — Apple Silicon에서 Qwen3.6-35B-A3B를 더 빠르게
  돌리는 Rust + Metal 추론 엔진" (alltoptrend.co.kr): §4 (three compute patterns:
  8 of 256 experts per token, uneven groups), §5-1 (groupwise-affine 4-bit
  weights, 64 weights per bf16 scale and bias; dequantised tile by tile inside
  the grouped GEMM with FP32 accumulation), §5-2 (routing histogram, prefix scan,
  scatter and block map in one GPU command buffer; expert GEMM ~90% of prefill;
  bounded chunks for long prompts).
* [C] "Apple silicon용 Lily, Qwen 추론 최적화" (aitrends.kr): section "Qwen 구조와
  Prefill 경로" (router picks 8 of 256 experts plus 1 shared expert), section
  "GPU 상주와 메모리 절감" (per-token expert selection, then histogram of
  allocations, prefix scan for start offsets, scatter of rows into expert
  groups), glossary entry on groupwise affine 4-bit quantisation.

What the pages leave open is fixed by the layer specification that accompanies
them (softmax over E, keep top-k, renormalise; SwiGLU expert FFN; shared expert
added with weight 1; packing 8 codes per uint32, low nibble first along K;
dequantised weight = bf16(fp32(scale)*q + fp32(bias)); SwiGLU activation rounded
to bf16 before the down projection). Readings taken where both are silent:

* top-k ranks experts by the fp32 logit (softmax is strictly increasing, so the
  order is the order of probabilities), ties to the lower expert index, ids of a
  token in descending order;
* rows of an expert group are in ascending (token, slot) order;
* gate/up rows: rows 0..f-1 of the [2f, d] matrix are the gate projection, rows
  f..2f-1 the up projection;
* block map: for each expert in ascending order, tiles of at most ``block_m``
  consecutive group rows, as (expert, first row, row count); empty experts get
  no tile; the shared expert is not part of the routing output;
* the combine accumulates in high precision and rounds y to bf16 once.

Arithmetic: float64 throughout except where the specification fixes a rounding
(bf16 weights, bf16 activation, fp32 routing weights, bf16 output).

Parity pins: every function here is pinned by ``tests/test_oracle_*.py``
against closed forms, hand-worked golden fixtures, library routines and brute
force; none is "parity unpinned".
"""
from __future__ import annotations

import dataclasses

import numpy as np

# --------------------------------------------------------------------------- bf16


def to_bf16(v) -> np.ndarray:
    """Round real values to bf16 (round to nearest, ties to even); returns uint16 bits.

    bf16 keeps 8 significant bits and the fp32 exponent range, so for
    v = m * 2**e with 0.5 <= |m| < 1 the rounding quantum is 2**(e-8), floored at
    the smallest subnormal 2**-133. Scaling by a power of two and ``np.round``
    (half to even) are exact in float64, so this is the correctly rounded value
    for any float64 input, with no double rounding through fp32.
    """
    v = np.asarray(v, dtype=np.float64)
    _, ex = np.frexp(v)
    q = np.maximum(ex - 8, -133)
    r = np.ldexp(np.round(np.ldexp(v, -q)), q)
    with np.errstate(over="ignore", invalid="ignore"):
        f32 = r.astype(np.float32)  # exact for every bf16 value; overflow -> inf
    bits = (f32.view(np.uint32) >> np.uint32(16)).astype(np.uint16)
    bits = np.where(np.isnan(v), np.uint16(0x7FC0), bits)
    return bits.astype(np.uint16)


def bf16_value(bits) -> np.ndarray:
    """Value of bf16 bit patterns, as float64 (exact)."""
    b = np.asarray(bits, dtype=np.uint16).astype(np.uint32) << np.uint32(16)
    with np.errstate(invalid="ignore"):
        return b.view(np.float32).astype(np.float64)


# ----------------------------------------------------------------- Q4 weight format


def unpack_codes(qw) -> np.ndarray:
    """4-bit codes from packed words: 8 codes per uint32, low nibble first along K.

    qw[..., K/8] uint32 -> codes[..., K] uint8 with code c = (qw[c // 8] >> 4*(c % 8)) & 15.
    Format: [A] §5-1 (4-bit groupwise-affine checkpoint).
    """
    qw = np.asarray(qw, dtype=np.uint32)
    shifts = (4 * np.arange(8, dtype=np.uint32))
    codes = (qw[..., :, None] >> shifts) & np.uint32(15)
    return codes.reshape(*qw.shape[:-1], qw.shape[-1] * 8).astype(np.uint8)


def pack_codes(codes) -> np.ndarray:
    """Inverse of :func:`unpack_codes` (used to build hand-made groups in tests)."""
    c = np.asarray(codes, dtype=np.uint32)
    c = c.reshape(*c.shape[:-1], c.shape[-1] // 8, 8)
    return np.bitwise_or.reduce(c << (4 * np.arange(8, dtype=np.uint32)), axis=-1).astype(np.uint32)


def dequant(qw, scale_bits, bias_bits) -> np.ndarray:
    """Groupwise-affine 4-bit dequantisation to bf16 values (returned as float64).

    Each group of 64 consecutive weights along K shares one bf16 scale and one
    bf16 bias ([A] §5-1; [C] glossary). The value of code q in group g is
    w = bf16( fp32(fp32(scale_g) * q) + fp32(bias_g) ): an fp32 multiply, an fp32
    add, then one rounding to bf16, as the layer specification defines it.

    qw [..., K/8] uint32, scale_bits/bias_bits [..., K/64] uint16 -> [..., K] float64.
    """
    q = unpack_codes(qw).astype(np.float32)
    K = q.shape[-1]
    s = np.repeat(bf16_value(scale_bits).astype(np.float32), 64, axis=-1)[..., :K]
    b = np.repeat(bf16_value(bias_bits).astype(np.float32), 64, axis=-1)[..., :K]
    prod = np.multiply(s, q, dtype=np.float32)
    tot = np.add(prod, b, dtype=np.float32)
    return bf16_value(to_bf16(tot.astype(np.float64)))


# ------------------------------------------------------------------------ routing


@dataclasses.dataclass
class Route:
    """Routing result for T tokens, E experts, top-k, block map tile ``block_m``.

    ids [T,k] int32    chosen experts, descending logit, ties to lower index
    w   [T,k] float32  renormalised softmax weights of the chosen experts
    counts  [E]        rows per expert (histogram)
    offsets [E+1]      exclusive prefix sum of counts; offsets[E] = T*k
    perm [T*k]         perm[offsets[e] + r] = t*k + j for the r-th (t, j) of e
    inv  [T*k]         inv[t*k + j] = position of (t, j) in perm
    tiles [n_tiles,3]  (expert, first row, rows) per tile of at most block_m rows
    """
    T: int
    E: int
    k: int
    block_m: int
    ids: np.ndarray
    w: np.ndarray
    counts: np.ndarray
    offsets: np.ndarray
    perm: np.ndarray
    inv: np.ndarray
    tiles: np.ndarray

    @property
    def n_tiles(self) -> int:
        return int(self.tiles.shape[0])


def max_tiles(T: int, E: int, k: int, block_m: int) -> int:
    """Upper bound on the block-map length: sum_e ceil(c_e/BM) <= T*k//BM + #non-empty."""
    return (T * k) // block_m + min(E, T * k)


def route(logits, k: int, block_m: int = 128) -> Route:
    """Expert selection, histogram, exclusive scan, scatter and block map.

    Step order from [C] "GPU 상주와 메모리 절감" (select per token, count with a
    histogram, prefix scan for start offsets, scatter rows into expert groups)
    and [A] §5-2 (plus the block map that drives the grouped GEMM). Weights:
    softmax over all E experts, keep the top k, renormalise to sum 1 (the layer
    specification), evaluated in float64 and rounded once to fp32.
    """
    L32 = np.asarray(logits, dtype=np.float32)
    if not np.all(np.isfinite(L32)):
        raise ValueError("router logits must be finite")
    T, E = L32.shape
    if not (1 <= k <= E):
        raise ValueError("need 1 <= k <= E")
    L = L32.astype(np.float64)
    # softmax over all E experts
    p = np.exp(L - L.max(axis=1, keepdims=True))
    p = p / p.sum(axis=1, keepdims=True)
    # selection: rank by logit descending; a stable sort keeps equal logits in
    # ascending expert order, which is the tie rule
    order = np.argsort(-L32, axis=1, kind="stable")
    ids = order[:, :k].astype(np.int32)
    psel = np.take_along_axis(p, ids.astype(np.int64), axis=1)
    w = (psel / psel.sum(axis=1, keepdims=True)).astype(np.float32)
    # histogram of allocations
    flat = ids.reshape(-1)
    counts = np.bincount(flat, minlength=E).astype(np.int32)
    # exclusive prefix scan -> start offsets
    offsets = np.zeros(E + 1, dtype=np.int64)
    offsets[1:] = np.cumsum(counts)
    # scatter: rows of each expert in ascending (t, j) order (stable sort by expert)
    perm = np.argsort(flat, kind="stable").astype(np.int32)
    inv = np.empty(T * k, dtype=np.int32)
    inv[perm] = np.arange(T * k, dtype=np.int32)
    # block map
    tiles = []
    for e in range(E):
        for s in range(0, int(counts[e]), block_m):
            tiles.append((e, int(offsets[e]) + s, min(block_m, int(counts[e]) - s)))
    tiles = np.array(tiles, dtype=np.int32).reshape(-1, 3)
    return Route(T, E, k, block_m, ids, w, counts, offsets.astype(np.int32), perm, inv, tiles)


def router_logits(x_bits, wr_bits) -> np.ndarray:
    """Router projection: logits[t, e] = sum_c x[t, c] * Wr[e, c].

    The router scores every expert for every token before the top-k choice
    ([C] "Qwen 구조와 Prefill 경로": 8 of 256 experts per token; "GPU 상주와 메모리
    절감": the selection stays on the GPU). x [T, d] and Wr [E, d] are bf16 bits;
    products of bf16 values accumulate in float64. Returns float64 [T, E].
    """
    X = bf16_value(np.asarray(x_bits))
    Wr = bf16_value(np.asarray(wr_bits))
    return X @ Wr.T


# ---------------------------------------------------------------------------- FFN


def silu(g):
    return g / (1.0 + np.exp(-g))


def _ffn_one(X, qgu, sgu, bgu, qdn, sdn, bdn, f):
    """One expert's SwiGLU FFN on the rows X (float64 values of bf16 inputs).

    gate/up: G, U = X Wg^T, X Wu^T with the dequantised [2f, d] matrix (rows
    0..f-1 gate, f..2f-1 up); a = bf16(silu(G) * U); out = a Wd^T with the
    dequantised [d, f] down matrix. Products of bf16 values accumulate in float64.
    """
    Wgu = dequant(qgu, sgu, bgu)
    G = X @ Wgu[:f].T
    U = X @ Wgu[f:].T
    A = bf16_value(to_bf16(silu(G) * U))
    Wd = dequant(qdn, sdn, bdn)
    return A @ Wd.T


def expert_ffn(x_bits, W, r: Route, tokens=None, return_acc=False, experts=None, shared=True):
    """Grouped expert FFN with weighted combine and the shared expert.

    For each expert e and each row of its group (token t, slot j):
    y_acc[t] += w[t, j] * FFN_e(x[t]); then the shared expert is added with
    weight 1 and y = bf16(y_acc). Expert groups and routing from [C] "Qwen 구조와
    Prefill 경로" (8 of 256 experts plus one shared expert); the 4-bit weights
    are expanded per expert with :func:`dequant` ([A] §5-1).

    ``tokens``: optional sorted token subset; rows of other tokens are skipped
    (the layer is independent per token). ``experts`` / ``shared``: restrict the
    work to some expert groups (used to time a bounded sample of the layer).
    Returns bf16 bits [len(tokens) or T, d].
    """
    x_bits = np.asarray(x_bits)
    T, d = x_bits.shape
    k, E = r.k, r.E
    tok_list = np.arange(T) if tokens is None else np.asarray(tokens, dtype=np.int64)
    where = -np.ones(T, dtype=np.int64)
    where[tok_list] = np.arange(len(tok_list))
    acc = np.zeros((len(tok_list), d), dtype=np.float64)
    X = bf16_value(x_bits)
    for e in (range(E) if experts is None else experts):
        rows = r.perm[r.offsets[e]:r.offsets[e + 1]].astype(np.int64)
        t, j = rows // k, rows % k
        keep = where[t] >= 0
        t, j = t[keep], j[keep]
        if t.size == 0:
            continue
        out = _ffn_one(X[t], W.gu_qw[e], W.gu_scale[e], W.gu_bias[e],
                       W.dn_qw[e], W.dn_scale[e], W.dn_bias[e], W.f)
        acc[where[t]] += r.w[t, j].astype(np.float64)[:, None] * out
    if W.f_s and shared:
        out = _ffn_one(X[tok_list], W.sgu_qw[0], W.sgu_scale[0], W.sgu_bias[0],
                       W.sdn_qw[0], W.sdn_scale[0], W.sdn_bias[0], W.f_s)
        acc += out
    y = to_bf16(acc)
    return (y, acc) if return_acc else y


def dense_moe(x_bits, W, ids, w, return_acc=False):
    """Brute-force MoE: run every expert on every token and combine with a mask.

    mask[t, e] = w[t, j] if ids[t, j] == e else 0; y_acc = sum_e mask[:, e] *
    FFN_e(x) in ascending e, plus the shared expert with weight 1. Uses no
    histogram, scan, permutation or block map, so it checks those steps.
    """
    X = bf16_value(np.asarray(x_bits))
    T, d = X.shape
    E = W.E
    mask = np.zeros((T, E), dtype=np.float64)
    for j in range(ids.shape[1]):
        mask[np.arange(T), ids[:, j]] = w[:, j].astype(np.float64)
    acc = np.zeros((T, d), dtype=np.float64)
    for e in range(E):
        out = _ffn_one(X, W.gu_qw[e], W.gu_scale[e], W.gu_bias[e],
                       W.dn_qw[e], W.dn_scale[e], W.dn_bias[e], W.f)
        acc += mask[:, e:e + 1] * out
    if W.f_s:
        acc += _ffn_one(X, W.sgu_qw[0], W.sgu_scale[0], W.sgu_bias[0],
                        W.sdn_qw[0], W.sdn_scale[0], W.sdn_bias[0], W.f_s)
    y = to_bf16(acc)
    return (y, acc) if return_acc else y


def moe_layer(x_bits, logits, W, k, block_m=128, tokens=None):
    """Routing followed by the expert FFN: (Route, y bf16 bits)."""
    r = route(logits, k, block_m)
    return r, expert_ffn(x_bits, W, r, tokens=tokens)


def rms_unit(y_bits, x_bits) -> np.ndarray:
    """Next layer's input in the chunked multi-layer run: bf16((y+x)/rms(y+x)) per token.

    Plainest reading of "previous output plus residual, rescaled to unit RMS
    per token": no epsilon, no learned gain. Bounded-chunk prefill: [A] §5-2,
    [C] "GPU 상주와 메모리 절감".
    """
    v = bf16_value(y_bits) + bf16_value(x_bits)
    rms = np.sqrt(np.mean(v * v, axis=-1, keepdims=True))
    return to_bf16(v / rms)

