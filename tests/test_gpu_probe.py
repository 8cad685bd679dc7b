"""tcgen05 building blocks in isolation: the MMA with both A placements, and the
in-register 4-bit dequantisation, against exact host results."""
import numpy as np
import pytest
import torch

import oracle as O
from routing_q4_grouped_gb300 import moeq4, synth
from gpu_helpers import bits, dev

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("a_tmem", [0, 1])
@pytest.mark.parametrize("N,K", [(16, 64), (128, 128), (256, 256), (48, 1024), (208, 192)])
def test_mma_exact_small_integers(a_tmem, N, K):
    # integer operands: every product and partial sum is exact in fp32, so D must be exact
    g = torch.Generator().manual_seed(N * 1000 + K + a_tmem)
    A = torch.randint(-4, 5, (128, K), generator=g).to(torch.bfloat16).cuda()
    B = torch.randint(-4, 5, (N, K), generator=g).to(torch.bfloat16).cuda()
    D = torch.full((128, N), float("nan"), device="cuda")
    moeq4.moe_debug_mma(bool(a_tmem), A, B, D)
    torch.cuda.synchronize()
    ref = A.double().cpu() @ B.double().cpu().T
    assert torch.equal(D.cpu().double(), ref)


@pytest.mark.parametrize("a_tmem", [0, 1])
def test_mma_random_bf16(a_tmem):
    g = torch.Generator().manual_seed(7)
    A = torch.randn((128, 512), generator=g).to(torch.bfloat16).cuda()
    B = torch.randn((96, 512), generator=g).to(torch.bfloat16).cuda()
    D = torch.empty((128, 96), device="cuda")
    moeq4.moe_debug_mma(bool(a_tmem), A, B, D)
    torch.cuda.synchronize()
    ref = A.double().cpu() @ B.double().cpu().T
    assert (D.cpu().double() - ref).abs().max() < 1e-3


def _dequant_gpu(qw, s, b):
    rows = qw.shape[0] * qw.shape[1] if qw.ndim == 3 else qw.shape[0]
    K = qw.shape[-1] * 8
    out = torch.empty((rows, K), dtype=torch.bfloat16, device="cuda")
    moeq4.moe_debug_dequant(dev(qw.reshape(rows, -1)), dev(s.reshape(rows, -1)),
                            dev(b.reshape(rows, -1)), out)
    torch.cuda.synchronize()
    return bits(out)


@pytest.mark.parametrize("name", ["tiny", "t512"])
def test_dequant_bit_exact(name):
    W = synth.gen_weights(synth.CONFIGS[name])
    E = min(W.E, 4)
    for qw, s, b in ((W.gu_qw[:E], W.gu_scale[:E], W.gu_bias[:E]),
                     (W.dn_qw[:E], W.dn_scale[:E], W.dn_bias[:E])):
        got = _dequant_gpu(qw, s, b)
        ref = O.to_bf16(O.dequant(qw, s, b)).reshape(got.shape)
        assert np.array_equal(got, ref)


def test_dequant_hand_groups():
    codes = np.tile(np.arange(16, dtype=np.uint8), 4)[None, :].repeat(4, 0)
    qw = O.pack_codes(codes)
    s = np.array([[0x3F80], [0x3B80], [0x0000], [0x3BA4]], np.uint16)
    b = np.array([[0x0000], [0xBD00], [0xC040], [0xBD1A]], np.uint16)
    got = _dequant_gpu(qw, s, b)
    assert np.array_equal(got, O.to_bf16(O.dequant(qw, s, b)))
    assert np.array_equal(O.bf16_value(got[0]), codes[0].astype(np.float64))


def test_dequant_scale_range():
    # scales from subnormal to 8 in magnitude, both signs, and zero: the
    # in-register expansion bit-exact against the oracle
    rng = np.random.default_rng(21)
    rows, K = 64, 512
    codes = rng.integers(0, 16, size=(rows, K), dtype=np.uint8)
    qw = O.pack_codes(codes)
    g = rows * K // 64
    expo = rng.integers(0, 131, size=g)                     # bf16 exponent field 0..130
    s = ((rng.integers(0, 2, size=g) << 15) | (expo << 7) | rng.integers(0, 128, size=g))
    s[:8] = [0x0000, 0x8000, 0x3E7F, 0x3E80, 0xBE7F, 0xBE80, 0x0001, 0x3F80]   # 2^-2 edges, subnormal
    b = O.to_bf16(rng.standard_normal(g) * 0.05)
    s = s.astype(np.uint16).reshape(rows, -1)
    b = np.asarray(b, np.uint16).reshape(rows, -1)
    got = _dequant_gpu(qw, s, b)
    assert np.array_equal(got, O.to_bf16(O.dequant(qw, s, b)).reshape(got.shape))


def test_tmem_16x256b_fragment_layout():
    """Thread t of warp q, repetition j: registers 4j, 4j+1 hold lane base + t/4 at
    columns 8j + 2(t%4) + {0, 1}; registers 4j+2, 4j+3 hold lane base + 8 + t/4."""
    out = torch.zeros((128, 32), dtype=torch.int32, device="cuda")
    moeq4.moe_debug_tmem_layout(out)
    torch.cuda.synchronize()
    got = out.cpu().numpy().astype(np.int64) & 0xFFFFFFFF
    want = np.zeros((128, 32), dtype=np.int64)
    for q in range(4):
        for t in range(32):
            for half in range(2):
                base = 32 * q + 16 * half
                for j in range(4):
                    for r in range(4):
                        lane = base + t // 4 + (8 if r >= 2 else 0)
                        col = 8 * j + 2 * (t % 4) + (r & 1)
                        want[32 * q + t, 16 * half + 4 * j + r] = (lane << 16) | col
    assert np.array_equal(got, want)


def _pack_reference(qw, scale, bias, kind, F_or_d):
    """The kernel-native layout, built from its description in include/moeq4.h."""
    E, R, W8 = qw.shape
    K = W8 * 8
    nch, units = K // 64, R // 256
    e, p, c, t, L = np.meshgrid(np.arange(E), np.arange(units), np.arange(nch), np.arange(2),
                                np.arange(128), indexing="ij")
    if kind == 0:
        row = ((L >> 3) & 1) * F_or_d + 64 * (2 * p + t) + 8 * (L >> 4) + (L & 7)
    else:
        row = 256 * p + 128 * t + L
    words = qw[e[..., None], row[..., None], c[..., None] * 8 + np.arange(8)]      # [..., 8]
    nib = (words[..., None] >> (4 * np.arange(8, dtype=np.uint32))) & 15          # [..., 8 words, 8 nibbles]
    order = np.array([0, 2, 4, 6, 1, 3, 5, 7])
    perm = np.bitwise_or.reduce(nib[..., order] << (4 * np.arange(8, dtype=np.uint32)), axis=-1)
    perm = perm.astype(np.uint32)
    halves = perm.reshape(E, units, nch, 2, 128, 2, 4)                              # [.., tile, row, half, 4]
    stored = halves.transpose(0, 1, 2, 3, 5, 4, 6)                                  # [.., tile, half, row, 4]
    codes = np.ascontiguousarray(stored).astype("<u4").view(np.uint8)
    codes = codes.reshape(E, units, nch, 2 * 128 * 32)
    g = row * nch + c
    sb = scale.reshape(E, -1)[e, g].astype(np.uint32) | (bias.reshape(E, -1)[e, g].astype(np.uint32) << 16)
    sb = sb.astype("<u4").reshape(E, units, nch, 256).view(np.uint8)
    return np.concatenate([codes, sb], axis=-1).reshape(-1)


def test_prepack_matches_documented_layout():
    import dataclasses
    cfg = dataclasses.replace(synth.CONFIGS["tiny"], f_s=256, f=256, d=512)
    W = synth.gen_weights(cfg)
    dw = moeq4.DeviceWeights.from_host(W)
    torch.cuda.synchronize()
    got = dw.packed.cpu().numpy()
    ref = np.concatenate([
        _pack_reference(W.gu_qw, W.gu_scale, W.gu_bias, 0, cfg.f),
        _pack_reference(W.dn_qw, W.dn_scale, W.dn_bias, 1, cfg.d),
        _pack_reference(W.sgu_qw, W.sgu_scale, W.sgu_bias, 0, cfg.f_s),
        _pack_reference(W.sdn_qw, W.sdn_scale, W.sdn_bias, 1, cfg.d)])
    assert got.shape == ref.shape
    assert np.array_equal(got, ref)


def test_l2_prefetch_leaves_data_and_errors_alone():
    t = torch.arange(1 << 20, dtype=torch.int32, device="cuda")
    before = t.clone()
    moeq4.moe_l2_prefetch(t)
    moeq4.moe_l2_prefetch(t, 4096 + 16)
    torch.cuda.synchronize()
    assert torch.equal(t, before)
    assert moeq4.lib().moe_l2_prefetch(None, 16, None) == -1            # MOE_ERR_ARG
