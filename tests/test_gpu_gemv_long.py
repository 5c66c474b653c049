"""The split-K GEMV on long K slices, against the oracle in the block layout.

Slices of many rows stream in 18 KB stages (64 rows of two blocks per
thread, or 128 rows of one) instead of 32-row ones, with their own ring
depth and warp groups.  These shapes take that path; each is compared with
the fp64 oracle (engine page §3.4) element by element at the stated
tolerance 1e-3 * sum|a*w| + 1e-6, in full or on seeded block columns.
"""

import numpy as np
import pytest

import oracle
import seeded_inputs as si
from gpu_util import assert_within_matmul_tol, device, to_dev, to_host64, torch

import quantized_weight_q4_gb300 as q4

pytestmark = pytest.mark.gpu


def run(A, B, M, N, K):
    C = torch.empty((M, N), dtype=torch.float32, device=device())
    q4.q4_matmul_ex(C, to_dev(A), to_dev(B), M, N, K)
    torch.cuda.synchronize()
    assert q4.q4_get_device_status() == q4.Q4_OK
    return to_host64(C)


@pytest.mark.parametrize("M,K,N,adt", [(1, 16384, 2048, "f32"), (2, 8192, 1024, "bf16"),
                                       (4, 8192, 512, "f32"), (1, 11008, 4096, "f32"),
                                       (3, 12000, 520, "bf16")])
def test_long_slices_full(M, K, N, adt):
    A = si.activations_bf16(M, K, seed=K) if adt == "bf16" else si.activations_f32(M, K, seed=K)
    B = si.q4_weights(K, N, seed=N)
    C = run(A, B, M, N, K)
    C64, S = oracle.matmul(A, B, M, N, K)
    assert_within_matmul_tol(C, C64, S, f"M={M} K={K} N={N}")


def test_16384_square_sampled_block_columns():
    """K = N = 16384 at M = 1: 24 seeded block columns (every row of K) against
    the oracle; the columns span first, last and interior column tiles."""
    M, K, N = 1, 16384, 16384
    A = si.activations_f32(M, K, seed=5)
    B = si.q4_weights(K, N, seed=5)
    C = run(A, B, M, N, K)
    nb = si.nblocks(N)
    cols = np.unique(np.concatenate([[0, nb - 1, 255, 256],
                                     si.rng(5, 6).choice(nb, size=20, replace=False)]))
    Bs = B.reshape(K, nb, 18)[:, cols].reshape(K, -1)
    C64, S = oracle.matmul(A, Bs, M, 32 * len(cols), K)
    got = C.reshape(M, nb, 32)[:, cols].reshape(M, -1)
    assert_within_matmul_tol(got, C64, S, "16384 x 16384 sampled")
