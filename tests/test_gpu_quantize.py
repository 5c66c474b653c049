"""GPU Q4_0 encoder against the oracle's encoder, byte for byte.

Codes are integers decided by floating point: both sides take every step as
one fp32 operation in the same order (no fused multiply-add), so the blocks
must be identical, scale bits included.
"""

import numpy as np
import pytest

import oracle
import seeded_inputs as si
from gpu_util import device, to_dev, torch

import quantized_weight_q4_gb300 as q4

pytestmark = pytest.mark.gpu


def quantize(W, K, N):
    B = torch.empty((K, si.nblocks(N) * 18), dtype=torch.uint8, device=device())
    q4.q4_quantize(B, to_dev(W), K, N)
    torch.cuda.synchronize()
    return B.cpu().numpy()


def weights(K, N, seed):
    W = (si.rng(seed, 1).standard_normal((K, N)) * 0.02).astype(np.float32)
    if K > 3:
        W[1] = 0.0                                   # a zero row
        n2 = N // 2
        W[2, 0:2 * n2:2] = -W[2, 1:2 * n2:2]        # equal magnitudes, opposite signs
        W[3, :16] = np.float32(-0.4375) * (1 + (np.arange(16) % 3))   # half steps
    return W


@pytest.mark.parametrize("K,N", [(1, 32), (3, 40), (37, 200), (64, 4096), (300, 1000), (9, 31)])
@pytest.mark.parametrize("bf16", [False, True])
def test_quantize_parity(K, N, bf16):
    W = weights(K, N, seed=K + N)
    if bf16:
        W = si.f32_to_bf16_bits(W)
    assert np.array_equal(quantize(W, K, N), oracle.quantize(W, K, N)), f"K={K} N={N} bf16={bf16}"


def test_quantize_large_and_overflowing_scales():
    K, N = 8, 256
    W = (si.rng(3, 1).standard_normal((K, N)) * 1e4).astype(np.float32)
    W[0, 0] = 6e5          # d = -75000: beyond fp16, stored as -inf
    W[1, 5] = -65504.0 * 8
    assert np.array_equal(quantize(W, K, N), oracle.quantize(W, K, N))


def test_quantize_full_matrix_round_trip():
    """A 5120 x 12288 matrix: blocks equal to the oracle's, and dequantising
    them on the GPU returns each weight within one step of its block (a full
    step where code 16 would be needed), widened by the fp16 rounding of the
    scale (relative 2^-11, times at most 8 steps)."""
    K, N = 5120, 12288
    W = weights(K, N, seed=1)
    B = quantize(W, K, N)
    assert np.array_equal(B, oracle.quantize(W, K, N))
    R = torch.empty((K, N), dtype=torch.float32, device=device())
    q4.q4_dequant(R, to_dev(B), K, N)
    torch.cuda.synchronize()
    R = R.cpu().numpy().astype(np.float64)
    d = np.abs(B.reshape(K, -1, 18)[:, :, :2].copy().view(np.float16).astype(np.float64))
    step = np.repeat(d[:, :, 0], 32, axis=1)[:, :N]
    assert (np.abs(R - W) <= step * (1 + 8 * 2.0 ** -11) * 1.0001 + 1e-9).all()
