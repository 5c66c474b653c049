"""GPU GEMV on planar Q4_0 weights (Q4_LAYOUT_PLANAR, q4_repack's layout).

The planar layout holds the same blocks as Q4_LAYOUT_BLOCKS, split into a
plane of fp16 scales d[K][nb] and a plane of nibbles qs[K][nb][16] that
starts at q4_planar_qs_offset(K, N).  The GEMV reads it with the same launch
shape and the same arithmetic, so every output must equal the block-layout
output bit for bit; the block-layout path is itself checked against the
oracle, and a few cases here are checked against the oracle directly.

The planar bytes are built on the host from the header's description of the
layout (not through q4_repack), so a repack mistake cannot hide a GEMV one.
"""

import numpy as np
import pytest

import oracle
import seeded_inputs as si
from gpu_util import assert_within_matmul_tol, device, to_dev, to_host64, torch

import quantized_weight_q4_gb300 as q4

pytestmark = pytest.mark.gpu


def planar_bytes(B, K, N):
    """Q4_LAYOUT_PLANAR bytes of the blocks B [K, nb*18]: the scales plane,
    zero bytes up to the nibble plane's offset, then the nibble plane."""
    nb = si.nblocks(N)
    blocks = B.reshape(K * nb, 18)
    off = q4.q4_planar_qs_offset(K, N)
    out = np.zeros(q4.q4_planar_bytes(K, N), dtype=np.uint8)
    out[:2 * K * nb] = blocks[:, :2].reshape(-1)
    out[off:off + 16 * K * nb] = blocks[:, 2:].reshape(-1)
    return out


def run(A, B, M, N, K, layout, c_dtype=torch.float32):
    C = torch.empty((M, N), dtype=c_dtype, device=device())
    q4.q4_matmul_ex(C, to_dev(A), to_dev(B), M, N, K, b_layout=layout)
    torch.cuda.synchronize()
    assert q4.q4_get_device_status() == q4.Q4_OK
    return C


def as_f32(A):
    """bf16 bits (uint16) widened exactly to fp32; fp32 unchanged."""
    if A.dtype == np.uint16:
        return (A.astype(np.uint32) << 16).view(np.float32)
    return A


def both_layouts(A, B, M, N, K, c_dtype=torch.float32):
    """The block layout with A widened to fp32 (so that it takes the GEMV at
    any M, with the same values of A) and the planar layout with A as given."""
    cb = run(as_f32(A), B, M, N, K, q4.Q4_LAYOUT_BLOCKS, c_dtype)
    cp = run(A, planar_bytes(B, K, N), M, N, K, q4.Q4_LAYOUT_PLANAR, c_dtype)
    return cb, cp


# (M, K, N): one to four rows (one chunk of 1, 2 or 4 rows, or three chunks of
# one), several chunks; ceil(N/32) a multiple of 8 (tensor copies) or not (the
# producer warp's copy); ragged N; K slices with a ragged last stage; K long
# enough for the 18 KB stages.
SHAPES = [(1, 1, 32), (1, 7, 40), (1, 100, 1000), (1, 4096, 4096), (1, 4096, 11008),
          (2, 333, 300), (3, 64, 96), (3, 1000, 2048), (4, 515, 800), (4, 1024, 4352),
          (5, 200, 520), (8, 300, 256), (17, 129, 1056), (64, 256, 512), (1, 16384, 2048),
          (2, 8192, 1024), (4, 4096, 2080)]


@pytest.mark.parametrize("M,K,N", SHAPES)
@pytest.mark.parametrize("adt", ["f32", "bf16"])
def test_planar_equals_blocks(M, K, N, adt):
    A = si.activations_f32(M, K, seed=M + K) if adt == "f32" else si.activations_bf16(M, K, seed=M + K)
    B = si.q4_weights(K, N, seed=N)
    cb, cp = both_layouts(A, B, M, N, K)
    assert torch.equal(cb, cp), f"planar != blocks for M={M} K={K} N={N} {adt}"


@pytest.mark.parametrize("M,K,N", [(1, 100, 1000), (3, 64, 96), (4, 515, 800), (17, 129, 1056),
                                   (1, 2048, 256)])
def test_planar_against_oracle(M, K, N):
    A = si.activations_f32(M, K, seed=3 * M + K)
    B = si.q4_weights(K, N, seed=N + 1)
    C = to_host64(run(A, planar_bytes(B, K, N), M, N, K, q4.Q4_LAYOUT_PLANAR))
    C64, S = oracle.matmul(A, B, M, N, K)
    assert_within_matmul_tol(C, C64, S, f"planar M={M} K={K} N={N}")


@pytest.mark.parametrize("K,N", [(9, 96), (300, 264), (1000, 4096)])
def test_planar_one_hot_rows_are_exact(K, N):
    B = si.q4_weights(K, N, seed=11)
    W = oracle.dequant_f32(B, K, N)
    P = planar_bytes(B, K, N)
    for k in sorted({0, K // 3, K - 1}):
        A = np.zeros((1, K), np.float32)
        A[0, k] = 1.0
        C = run(A, P, 1, N, K, q4.Q4_LAYOUT_PLANAR).cpu().numpy()
        assert np.array_equal(C[0], W[k]), k


@pytest.mark.parametrize("K,N", [(50, 40), (700, 1000), (64, 33)])
def test_planar_padding_never_contributes(K, N):
    A = si.activations_f32(3, K, seed=5)
    B = si.q4_weights(K, N, seed=5)
    Br = si.randomise_padding(B, K, N, 5, 6)
    assert torch.equal(run(A, planar_bytes(B, K, N), 3, N, K, q4.Q4_LAYOUT_PLANAR),
                       run(A, planar_bytes(Br, K, N), 3, N, K, q4.Q4_LAYOUT_PLANAR))


def test_planar_bf16_output_and_repack_input():
    """bf16 C equals the block layout's bf16 C; planar bytes made on the GPU by
    q4_repack give the same result as the host-built ones."""
    M, K, N = 2, 1000, 2048
    A = si.activations_bf16(M, K, seed=3)
    B = si.q4_weights(K, N, seed=3)
    cb, cp = both_layouts(A, B, M, N, K, c_dtype=torch.bfloat16)
    assert torch.equal(cb.view(torch.int16), cp.view(torch.int16))
    P = torch.zeros(q4.q4_planar_bytes(K, N), dtype=torch.uint8, device=device())
    q4.q4_repack(P, to_dev(B), K, N)
    C = torch.empty((M, N), dtype=torch.bfloat16, device=device())
    q4.q4_matmul_ex(C, to_dev(A), P, M, N, K, b_layout=q4.Q4_LAYOUT_PLANAR)
    torch.cuda.synchronize()
    assert torch.equal(C.view(torch.int16), cp.view(torch.int16))


@pytest.mark.parametrize("M", [1, 4])
def test_planar_large_equals_blocks(M):
    """K = 5120, N = 12288 (the batched decode shape), bf16 A: bit-identical to
    the block layout; and K = N = 16384 at M = 1 (18 KB stages)."""
    for K, N in ((5120, 12288), (16384, 16384)):
        if M > 1 and K == 16384:
            continue
        A = si.activations_bf16(M, K, seed=8 + M)
        B = si.q4_weights(K, N, seed=8)
        cb, cp = both_layouts(A, B, M, N, K)
        assert torch.equal(cb, cp), (M, K, N)


@pytest.mark.parametrize("M,K,N", [(65, 300, 520), (130, 1024, 4352)])
def test_planar_many_rows(M, K, N):
    """More than 64 rows (fp32 A): the GEMV in chunks of 4 rows, bit-identical
    to the block layout and within the oracle's tolerance."""
    A = si.activations_f32(M, K, seed=M)
    B = si.q4_weights(K, N, seed=M)
    cb, cp = both_layouts(A, B, M, N, K)
    assert torch.equal(cb, cp), (M, K, N)
    C64, S = oracle.matmul(A, B, M, N, K)
    assert_within_matmul_tol(to_host64(cp), C64, S, f"planar M={M}")
