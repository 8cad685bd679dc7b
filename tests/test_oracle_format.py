"""Pins for the oracle's bf16 rounding, nibble packing and 4-bit dequantisation."""
import json
import os

import numpy as np
import pytest
import torch

import oracle as O
from routing_q4_grouped_gb300 import synth

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


# ------------------------------------------------------------------ bf16 rounding

def test_bf16_hand_values():
    cases = {
        1.0: 0x3F80,
        -2.5: 0xC020,
        0.0: 0x0000,
        1.0 + 2.0 ** -8: 0x3F80,          # exact tie, even neighbour is 1.0
        1.0 + 3 * 2.0 ** -8: 0x3F82,      # exact tie, rounds up to even mantissa 2
        1.0 + 2.0 ** -8 + 2.0 ** -40: 0x3F81,  # just above the tie: up (no double rounding)
        2.0 ** -133: 0x0001,              # smallest bf16 subnormal
        float("inf"): 0x7F80,
    }
    for v, bits in cases.items():
        assert int(O.to_bf16(v)) == bits, (v, hex(int(O.to_bf16(v))), hex(bits))
    assert int(O.to_bf16(float("nan"))) & 0x7F80 == 0x7F80


def test_bf16_matches_torch_on_fp32_inputs():
    # any fp32 value is exact in float64, so the oracle must agree with the
    # library's fp32 -> bf16 round-to-nearest-even conversion bit for bit
    rng = np.random.default_rng(0)
    bits = rng.integers(0, 2 ** 32, size=200000, dtype=np.uint64).astype(np.uint32)
    v = bits.view(np.float32)
    v = v[np.isfinite(v)]
    v = np.concatenate([v, rng.standard_normal(50000).astype(np.float32),
                        (rng.standard_normal(1000) * 1e-39).astype(np.float32)])
    ref = torch.from_numpy(v).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    got = O.to_bf16(v.astype(np.float64))
    assert np.array_equal(got, ref)


def test_bf16_value_roundtrip():
    b = np.arange(0, 1 << 16, dtype=np.uint32).astype(np.uint16)
    v = O.bf16_value(b)
    fin = np.isfinite(v)
    assert np.array_equal(O.to_bf16(v[fin]), b[fin])


# --------------------------------------------------------------------- packing

def test_unpack_hand_words():
    assert O.unpack_codes(np.array([0x76543210], dtype=np.uint32)).tolist() == list(range(8))
    assert O.unpack_codes(np.array([0xFEDCBA98], dtype=np.uint32)).tolist() == list(range(8, 16))
    # K index c lives in word c//8 at bit 4*(c%8)
    w = np.zeros(4, dtype=np.uint32)
    w[2] = np.uint32(0xA) << np.uint32(4 * 5)
    codes = O.unpack_codes(w)
    assert codes[2 * 8 + 5] == 10 and codes.sum() == 10


def test_pack_unpack_roundtrip():
    rng = np.random.default_rng(1)
    codes = rng.integers(0, 16, size=(7, 3, 128)).astype(np.uint8)
    assert np.array_equal(O.unpack_codes(O.pack_codes(codes)), codes)
    words = rng.integers(0, 2 ** 32, size=(5, 16), dtype=np.uint64).astype(np.uint32)
    assert np.array_equal(O.pack_codes(O.unpack_codes(words)), words)


# ------------------------------------------------------------------ dequant

def _group(codes, s_bits, b_bits):
    qw = O.pack_codes(np.asarray(codes, dtype=np.uint8))
    return O.dequant(qw, np.array([s_bits], np.uint16), np.array([b_bits], np.uint16))


def test_dequant_identity_scale():
    codes = np.arange(64) % 16
    w = _group(codes, 0x3F80, 0x0000)      # scale 1, bias 0 -> w = q
    assert np.array_equal(w, codes.astype(np.float64))


def test_dequant_power_of_two_affine():
    codes = np.arange(64) % 16
    # scale 2^-8 (0x3B80), bias -8 * 2^-8 = -2^-5 (0xBD00) -> (q - 8) / 256 exactly
    w = _group(codes, 0x3B80, 0xBD00)
    assert np.array_equal(w, (codes - 8) / 256.0)


def test_dequant_bias_only():
    codes = np.arange(64) % 16
    w = _group(codes, 0x0000, 0xC040)      # scale 0 -> every weight equals the bias (-3)
    assert np.all(w == -3.0)


def test_dequant_golden_group():
    g = json.load(open(os.path.join(GOLDEN, "dequant_group.json")))
    s, b = int(g["scale_bits"], 16), int(g["bias_bits"], 16)
    codes = np.arange(64) % 16
    w = _group(codes, s, b)
    for q, bits in g["expected"].items():
        assert int(O.to_bf16(w[int(q)])) == int(bits, 16), q


def test_dequant_group_boundaries():
    # K = 192: three groups with distinct scales; index 63 uses group 0, 64 group 1
    codes = np.full(192, 3, dtype=np.uint8)
    qw = O.pack_codes(codes)
    s = np.array([0x3F80, 0x4000, 0x4040], np.uint16)   # 1, 2, 3
    b = np.zeros(3, np.uint16)
    w = O.dequant(qw, s, b)
    assert w[0] == 3 and w[63] == 3 and w[64] == 6 and w[127] == 6 and w[128] == 9 and w[191] == 9


@pytest.mark.parametrize("name", ["tiny", "t512"])
def test_convention_equals_single_rounding(name):
    """fp32 multiply + fp32 add + bf16 rounding == one correctly rounded bf16(s*q+b).

    s*q + b is exact in float64 for bf16 s, b and q < 16, so to_bf16 of it is the
    single rounding that a fused bf16 multiply-add gives. Checked exhaustively
    over the 16 codes of every distinct (scale, bias) pair in the generated
    weights: this is what lets a kernel dequantise with one fused bf16 FMA.
    """
    cfg = synth.CONFIGS[name]
    W = synth.gen_weights(cfg)
    pairs = []
    for s, b in ((W.gu_scale, W.gu_bias), (W.dn_scale, W.dn_bias)):
        pairs.append((s.astype(np.uint32) << 16) | b.astype(np.uint32))
    if W.f_s:
        pairs.append((W.sgu_scale.astype(np.uint32) << 16) | W.sgu_bias.astype(np.uint32))
        pairs.append((W.sdn_scale.astype(np.uint32) << 16) | W.sdn_bias.astype(np.uint32))
    u = np.unique(np.concatenate([p.ravel() for p in pairs]))
    s_bits = (u >> 16).astype(np.uint16)
    b_bits = (u & 0xFFFF).astype(np.uint16)
    q = np.arange(16, dtype=np.float64)
    exact = O.bf16_value(s_bits)[:, None] * q[None, :] + O.bf16_value(b_bits)[:, None]
    single = O.to_bf16(exact)
    codes = np.tile(np.arange(16, dtype=np.uint8), 4)[None, :].repeat(len(u), 0)
    conv = O.to_bf16(O.dequant(O.pack_codes(codes), s_bits[:, None], b_bits[:, None]))[:, :16]
    assert np.array_equal(conv, single)


def test_synth_value_recipe():
    cfg = synth.CONFIGS["tiny"]
    W = synth.gen_weights(cfg)
    s = O.bf16_value(W.gu_scale)
    assert s.min() >= 0.0039 and s.max() <= 0.0081
    b = O.bf16_value(W.gu_bias)
    assert abs(np.mean(b + 7.5 * s)) < 2e-4 and np.std(b + 7.5 * s) < 0.002
    codes = O.unpack_codes(W.gu_qw)
    hist = np.bincount(codes.ravel(), minlength=16) / codes.size
    assert np.all(np.abs(hist - 1 / 16) < 0.005)
    x = O.bf16_value(synth.gen_x(cfg))
    assert abs(x.mean()) < 0.02 and abs(x.std() - 1) < 0.02
