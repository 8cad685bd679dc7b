"""Pins for the oracle's expert FFN, combine, shared expert and chunked-layer step."""
import dataclasses

import numpy as np
import pytest
import torch

import oracle as O
from routing_q4_grouped_gb300 import synth


def _const_weights(E, d, f, f_s, cg, cu, cd, scg=None, scu=None, scd=None):
    """Weights whose dequantised value is a per-(expert, matrix) constant.

    scale = 0 and bias = c give w = bf16(0*q + c) = c for every code.
    """
    def mat(ex, rows, K, consts_top, consts_bottom=None):
        qw = np.full((ex, rows, K // 8), 0x9A5C3E71, dtype=np.uint32)  # arbitrary codes
        s = np.zeros((ex, rows, K // 64), np.uint16)
        b = np.zeros((ex, rows, K // 64), np.uint16)
        for e in range(ex):
            if consts_bottom is None:
                b[e] = O.to_bf16(consts_top[e])
            else:
                b[e, : rows // 2] = O.to_bf16(consts_top[e])
                b[e, rows // 2:] = O.to_bf16(consts_bottom[e])
        return qw, s, b

    gu = mat(E, 2 * f, d, cg, cu)
    dn = mat(E, d, f, cd)
    kw = {}
    if f_s:
        sgu = mat(1, 2 * f_s, d, [scg], [scu])
        sdn = mat(1, d, f_s, [scd])
        kw = dict(sgu_qw=sgu[0], sgu_scale=sgu[1], sgu_bias=sgu[2],
                  sdn_qw=sdn[0], sdn_scale=sdn[1], sdn_bias=sdn[2])
    return synth.Q4Weights(E, d, f, f_s, gu[0], gu[1], gu[2], dn[0], dn[1], dn[2], **kw)


@pytest.mark.parametrize("f_s", [0, 128])
def test_closed_form_constant_weights(f_s):
    """All weights of a matrix equal one constant: y has a closed form.

    Gate, up and down constants differ per expert (and from the shared expert),
    so a swapped gate/up half, a wrong expert index or a dropped shared term
    changes the answer. For token t with sx = sum_c x[t,c]:
    g = cg*sx, u = cu*sx for every feature, a = bf16(silu(g)*u),
    each output feature = cd * f * a, y = bf16(sum_j w_j * that + shared term).
    """
    T, d, E, k, f = 16, 128, 4, 2, 64
    cg = [0.015625, -0.03125, 0.0234375, 0.0078125]
    cu = [0.0625, 0.046875, -0.0546875, 0.109375]
    cd = [0.25, -0.125, 0.375, 0.0625]
    W = _const_weights(E, d, f, f_s, cg, cu, cd, 0.01171875, -0.02734375, 0.1875)
    x = synth.to_bf16_bits(np.random.default_rng(0).standard_normal((T, d)))
    logits = np.random.default_rng(1).standard_normal((T, E)).astype(np.float32)
    r = O.route(logits, k, 8)
    y = O.expert_ffn(x, W, r)
    X = O.bf16_value(x)
    sx = X.sum(1)
    want = np.zeros(T)
    for t in range(T):
        for j in range(k):
            e = r.ids[t, j]
            g, u = cg[e] * sx[t], cu[e] * sx[t]
            a = O.bf16_value(O.to_bf16(g / (1 + np.exp(-g)) * u))
            want[t] += float(r.w[t, j]) * cd[e] * f * a
        if f_s:
            g, u = 0.01171875 * sx[t], -0.02734375 * sx[t]
            a = O.bf16_value(O.to_bf16(g / (1 + np.exp(-g)) * u))
            want[t] += 0.1875 * f_s * a
    assert np.array_equal(y, np.repeat(O.to_bf16(want)[:, None], d, 1))


def test_textbook_mlp_single_expert():
    """E = k = 1 without a shared expert is a plain SwiGLU MLP; compare with torch ops.

    The reference here dequantises with float64 torch arithmetic and rounds with
    torch's bf16 conversion, then uses torch.nn.functional.silu and matmul.
    """
    cfg = dataclasses.replace(synth.CONFIGS["tiny"], E=1, k=1, f=64, d=64)
    W = synth.gen_weights(cfg)
    T = 24
    x = synth.gen_x(cfg, T)
    r = O.route(np.zeros((T, 1), np.float32), 1, 16)
    y = O.expert_ffn(x, W, r)

    def deq(qw, s, b):
        qw = torch.from_numpy(qw.astype(np.int64))
        codes = torch.stack([(qw >> (4 * i)) & 15 for i in range(8)], -1).flatten(-2).double()
        sv = torch.from_numpy(s.astype(np.int32)).mul(65536).int().view(torch.float32).double()
        bv = torch.from_numpy(b.astype(np.int32)).mul(65536).int().view(torch.float32).double()
        return (sv.repeat_interleave(64, -1) * codes + bv.repeat_interleave(64, -1)) \
            .to(torch.bfloat16).double()

    Wgu = deq(W.gu_qw[0], W.gu_scale[0], W.gu_bias[0])
    Wd = deq(W.dn_qw[0], W.dn_scale[0], W.dn_bias[0])
    X = torch.from_numpy(x.astype(np.int32)).mul(65536).int().view(torch.float32).double()
    G, U = X @ Wgu[: cfg.f].T, X @ Wgu[cfg.f:].T
    A = (torch.nn.functional.silu(G) * U).float().to(torch.bfloat16).double()
    ref = (A @ Wd.T).float().to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    # torch rounds float64 through fp32 twice above; allow one bf16 ulp where that differs
    diff = np.abs(y.astype(np.int32) - ref.astype(np.int32))
    assert diff.max() <= 1 and (diff == 0).mean() > 0.99


@pytest.mark.parametrize("f_s", [0, 128])
def test_sparse_equals_dense_brute_force(f_s):
    cfg = dataclasses.replace(synth.CONFIGS["tiny"], f_s=f_s, T=48)
    W = synth.gen_weights(cfg)
    x = synth.gen_x(cfg)
    logits = synth.gen_logits(cfg)
    r = O.route(logits, cfg.k, 16)
    y, acc = O.expert_ffn(x, W, r, return_acc=True)
    yd, accd = O.dense_moe(x, W, r.ids, r.w, return_acc=True)
    assert np.allclose(acc, accd, rtol=1e-12, atol=1e-14)
    assert np.array_equal(y, yd)


def test_token_subset_matches_full():
    cfg = synth.CONFIGS["tiny"]
    W = synth.gen_weights(cfg)
    x = synth.gen_x(cfg)
    r = O.route(synth.gen_logits(cfg), cfg.k, 16)
    y = O.expert_ffn(x, W, r)
    sub = np.array([0, 5, 17, 63])
    assert np.array_equal(O.expert_ffn(x, W, r, tokens=sub), y[sub])


def test_rms_unit_closed_form():
    d = 64
    y = np.zeros((2, d), np.uint16)
    x = np.stack([O.to_bf16(np.full(d, 3.0)), O.to_bf16(np.full(d, -0.5))])
    out = O.rms_unit(y, x)
    assert np.all(out[0] == 0x3F80) and np.all(out[1] == 0xBF80)
    # alternating +a, -3a: mean square 5a^2 -> +1/sqrt(5), -3/sqrt(5)
    v = np.tile([1.0, -3.0], d // 2)
    out = O.rms_unit(np.zeros((1, d), np.uint16), O.to_bf16(v)[None])
    assert np.array_equal(out[0], O.to_bf16(v / np.sqrt(5.0)))


def test_process_pool_layer_equals_the_oracle():
    # the benchmark's CPU baseline spreads expert groups over processes; the
    # layer it computes is the oracle's
    from oracle.pool import OraclePool

    cfg = dataclasses.replace(synth.CONFIGS["tiny"], f_s=128)
    W = synth.gen_weights(cfg)
    x = synth.gen_x(cfg)
    logits = synth.gen_logits(cfg)
    pool = OraclePool(2)
    try:
        pool.load(W, x)
        r, y = pool.layer(logits, cfg.k, 16)
    finally:
        pool.close()
    ref = O.expert_ffn(x, W, O.route(logits, cfg.k, 16))
    assert np.array_equal(y, ref)
    assert r.n_tiles > 0
