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
