"""GPU dequantisation and repack, bit-exact against the hand-built golden blocks
and the fp64 oracle (C++ DeepSeek engine page, §2.2 block_q4_0 / dequantize)."""

import numpy as np
import pytest

import oracle
import seeded_inputs as si
from gpu_util import device, same_bf16, same_f32, to_dev, torch
from test_oracle_pins import _golden_blocks

import quantized_weight_q4_gb300 as q4

pytestmark = pytest.mark.gpu


def _gpu_dequant(B, K, N, bf16=False):
    Bd = to_dev(B)
    if bf16:
        W = torch.empty((K, N), dtype=torch.int16, device=device())
        q4.q4_dequant_bf16(W, Bd, K, N)
        torch.cuda.synchronize()
        return W.cpu().numpy().view(np.uint16)
    W = torch.empty((K, N), dtype=torch.float32, device=device())
    q4.q4_dequant(W, Bd, K, N)
    torch.cuda.synchronize()
    return W.cpu().numpy()


def test_golden_blocks_on_gpu():
    recs = _golden_blocks()
    B = np.stack([np.frombuffer(blk, np.uint8) for _, blk, _ in recs])   # K = #blocks, N = 32
    W = _gpu_dequant(B, len(recs), 32)
    for i, (name, _, vals) in enumerate(recs):
        assert same_f32(W[i], np.array(vals, np.float32)), name
        # signs of zeros too
        z = np.array(vals) == 0
        assert np.array_equal(np.signbit(W[i][z]), np.signbit(np.array(vals)[z])), name


@pytest.mark.parametrize("K,N", [(1, 1), (1, 32), (3, 40), (17, 1000), (64, 4096), (5, 12288)])
def test_dequant_bit_exact(K, N):
    B = si.q4_weights(K, N, seed=K + N, d_lo=-30.0, d_hi=30.0)
    assert same_f32(_gpu_dequant(B, K, N), oracle.dequant_f32(B, K, N))
    assert same_bf16(_gpu_dequant(B, K, N, bf16=True), oracle.dequant_bf16(B, K, N))


def test_dequant_every_scale_code():
    """All 65536 fp16 scale codes (including subnormals, Inf, NaN) x all codes q."""
    K = 65536 // 8
    B = np.zeros((K, 8, 18), np.uint8)
    codes = np.arange(65536, dtype=np.uint32).astype(np.uint16).reshape(K, 8)
    B[:, :, 0:2] = codes.view(np.uint8).reshape(K, 8, 2)
    ramp = np.array([0x10, 0x32, 0x54, 0x76, 0x98, 0xBA, 0xDC, 0xFE] * 2, np.uint8)
    B[:, :, 2:] = ramp
    B = B.reshape(K, 8 * 18)
    assert same_f32(_gpu_dequant(B, K, 256), oracle.dequant_f32(B, K, 256))
    assert same_bf16(_gpu_dequant(B, K, 256, bf16=True), oracle.dequant_bf16(B, K, 256))


@pytest.mark.parametrize("K,N", [(1, 32), (3, 40), (33, 1000), (128, 4096)])
def test_repack_round_trip(K, N):
    B = si.q4_weights(K, N, seed=9, d_lo=-5.0, d_hi=5.0)
    B = si.randomise_padding(B, K, N, 9, 5)   # padding bytes survive too
    nb = si.nblocks(N)
    Bd = to_dev(B)
    P = torch.zeros(q4.q4_planar_bytes(K, N), dtype=torch.uint8, device=device())
    q4.q4_repack(P, Bd, K, N)
    R = torch.zeros_like(Bd)
    q4.q4_unpack(R, P, K, N)
    torch.cuda.synchronize()
    assert np.array_equal(R.cpu().numpy(), B)
    # the planar layout is the scales plane, then the nibble plane
    p = P.cpu().numpy()
    blocks = B.reshape(K * nb, 18)
    off = q4.q4_planar_qs_offset(K, N)
    assert np.array_equal(p[:2 * K * nb].reshape(K * nb, 2), blocks[:, :2])
    assert np.array_equal(p[off:off + 16 * K * nb].reshape(K * nb, 16), blocks[:, 2:])
