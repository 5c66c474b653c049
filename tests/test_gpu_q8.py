"""GPU GEMV on Q8_0 weights (Q4_LAYOUT_Q8_0) against the oracle's Q8_0 matmul.

Tolerance as for Q4_0: |gpu - oracle| <= 1e-3 * sum_k |a*w| + 1e-6 per output
element.  Exact cases (one-hot A, padding, zeros, determinism) are compared
bit for bit.
"""

import numpy as np
import pytest

import oracle
import seeded_inputs as si
from gpu_util import assert_within_matmul_tol, device, to_dev, to_host64, torch

import quantized_weight_q4_gb300 as q4

pytestmark = pytest.mark.gpu


def run(A, B, M, N, K, c_dtype=torch.float32):
    C = torch.empty((M, N), dtype=c_dtype, device=device())
    q4.q4_matmul_ex(C, to_dev(A), to_dev(B), M, N, K, b_layout=q4.Q4_LAYOUT_Q8_0)
    torch.cuda.synchronize()
    return C


SHAPES = [(1, 1, 32), (1, 7, 40), (1, 100, 1000), (1, 4096, 4096), (2, 333, 300),
          (3, 64, 96), (4, 515, 800), (4, 1024, 4352), (5, 200, 520), (8, 300, 256),
          (17, 129, 1056), (64, 256, 512)]


@pytest.mark.parametrize("M,K,N", SHAPES)
@pytest.mark.parametrize("adt", ["f32", "bf16"])
def test_q8_parity(M, K, N, adt):
    A = si.activations_f32(M, K, seed=M + K) if adt == "f32" else si.activations_bf16(M, K, seed=M + K)
    B = si.q8_weights(K, N, seed=N)
    C = to_host64(run(A, B, M, N, K))
    C64, S = oracle.q8_matmul(A, B, M, N, K)
    assert_within_matmul_tol(C, C64, S, f"Q8_0 M={M} K={K} N={N} {adt}")


@pytest.mark.parametrize("K,N", [(9, 96), (300, 256), (1000, 4096), (64, 40)])
def test_q8_one_hot_rows_are_exact(K, N):
    B = si.q8_weights(K, N, seed=11)
    W = oracle.q8_dequant_f32(B, K, N)
    for k in sorted({0, K // 3, K - 1}):
        A = np.zeros((1, K), np.float32)
        A[0, k] = 1.0
        C = run(A, B, 1, N, K).cpu().numpy()
        assert np.array_equal(C[0], W[k]), k


@pytest.mark.parametrize("K,N", [(50, 40), (700, 1000), (64, 33)])
def test_q8_padding_never_contributes(K, N):
    A = si.activations_f32(3, K, seed=5)
    B = si.q8_weights(K, N, seed=5)
    Br = B.copy().reshape(K, -1, 34)
    first = N - (Br.shape[1] - 1) * 32
    Br[:, -1, 2 + first:] = si.rng(5, 99).integers(0, 256, size=(K, 32 - first), dtype=np.uint8)
    assert np.array_equal(run(A, B, 3, N, K).cpu().numpy(),
                          run(A, Br.reshape(K, -1), 3, N, K).cpu().numpy())


def test_q8_zero_scales_and_zero_activations():
    K, N = 200, 512
    B = si.q8_weights(K, N, seed=2).reshape(K, -1, 34).copy()
    B[:, :, :2] = 0
    A = si.activations_f32(2, K, seed=2)
    assert not run(A, B.reshape(K, -1), 2, N, K).any()
    assert not run(np.zeros((2, K), np.float32), si.q8_weights(K, N, seed=3), 2, N, K).any()


def test_q8_extreme_codes():
    """Codes -128 and 127 everywhere, both signs of d: exact small sums."""
    K, N = 64, 256
    B = si.q8_weights(K, N, seed=4).reshape(K, -1, 34).copy()
    B[:, :, 2:18] = 0x80
    B[:, :, 18:] = 0x7F
    A = si.activations_f32(1, K, seed=4)
    C = to_host64(run(A, B.reshape(K, -1), 1, N, K))
    C64, S = oracle.q8_matmul(A, B.reshape(K, -1), 1, N, K)
    assert_within_matmul_tol(C, C64, S, "extreme codes")


def test_q8_bf16_output_is_rounded_fp32():
    M, K, N = 2, 1000, 2048
    A = si.activations_bf16(M, K, seed=3)
    B = si.q8_weights(K, N, seed=3)
    C32 = run(A, B, M, N, K)
    C16 = run(A, B, M, N, K, c_dtype=torch.bfloat16)
    assert torch.equal(C32.to(torch.bfloat16).view(torch.int16), C16.view(torch.int16))


def test_q8_deterministic_and_large_sampled():
    """K = 5120, N = 12288 (the batched decode shape), M = 1 and 4: two runs
    are bit-identical, and 24 sampled block columns match the oracle."""
    K, N = 5120, 12288
    B = si.q8_weights(K, N, seed=8)
    for M in (1, 4):
        A = si.activations_bf16(M, K, seed=8 + M)
        c1 = run(A, B, M, N, K)
        c2 = run(A, B, M, N, K)
        assert torch.equal(c1, c2)
        cols = si.rng(M, 3).choice(N // 32, size=24, replace=False)
        Bs = B.reshape(K, -1, 34)[:, cols].reshape(K, -1)
        C64, S = oracle.q8_matmul(A, Bs, M, 24 * 32, K)
        got = to_host64(c1).reshape(M, -1, 32)[:, cols].reshape(M, -1)
        assert_within_matmul_tol(got, C64, S, f"Q8_0 5120x12288 M={M} sampled")


@pytest.mark.parametrize("M,K,N,adt", [(65, 300, 520, "f32"), (130, 1000, 256, "bf16"),
                                       (300, 129, 1056, "f32")])
def test_q8_many_rows(M, K, N, adt):
    """More than 64 rows: the GEMV in chunks of 4 rows (the last chunk
    ragged), every output against the oracle."""
    A = si.activations_f32(M, K, seed=M) if adt == "f32" else si.activations_bf16(M, K, seed=M)
    B = si.q8_weights(K, N, seed=M + 1)
    C = to_host64(run(A, B, M, N, K))
    C64, S = oracle.q8_matmul(A, B, M, N, K)
    assert_within_matmul_tol(C, C64, S, f"Q8_0 M={M} K={K} N={N} {adt}")
