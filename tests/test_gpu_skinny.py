"""The few-row tensor-core GEMM (bf16 A, 1 <= M <= 32): dequantised weights as
the MMA's A operand (128 output columns per instruction), tokens as its N
(16 or 32); q4_matmul_bf16_tiles takes it up to 32 rows and the split forms
above, which these cases also reach (M = 33 .. 64).  The engine page batches the tokens of a prompt into one
matmul (§5.2); with a few tokens the weights' bytes set the time.

Its product is A . bf16_rn(W) with fp32 accumulation, so parity is checked
against oracle.matmul_bf16_tiles within 1e-4 * sum|a * bf16(w)| + 1e-6, and
against A . W within the bf16 rounding bound.  One-hot rows reproduce the
bf16 tile values bit for bit, which pins the operand layouts, the
descriptors and the tile's column order.
"""

import numpy as np
import pytest

import oracle
import seeded_inputs as si
from gpu_util import assert_within_matmul_tol, device, to_dev, to_host64, torch

import quantized_weight_q4_gb300 as q4

pytestmark = pytest.mark.gpu


def tiles(A, B, M, N, K, c_dtype=torch.float32, workspace=None, stream=None):
    C = torch.empty((M, N), dtype=c_dtype, device=device())
    q4.q4_matmul_bf16_tiles(C, to_dev(A), to_dev(B), M, N, K, workspace=workspace, stream=stream)
    torch.cuda.synchronize()
    assert q4.q4_get_device_status() == q4.Q4_OK
    return C


def check_tiles(C, A, B, M, N, K, what):
    got = to_host64(C)
    Cb, Sb = oracle.matmul_bf16_tiles(A, B, M, N, K)
    err = np.abs(got - Cb)
    bad = ~(err <= 1e-4 * Sb + 1e-6)
    assert not bad.any(), f"{what}: {bad.sum()} beyond the bf16-tile tolerance"
    C64, S = oracle.matmul(A, B, M, N, K)
    assert (np.abs(got - C64) <= (2.0 ** -8 + 1e-4) * S + 1e-6).all(), what


# (M, K, N): every token tile (16, 32, 64) with M tails; K tails of the
# 128-row stage and of its 64-row halves (K = 8, 72, 520); N tails inside a
# 256-column tile (N = 250, 1000); the batched decode shape
CASES = [(1, 1024, 256), (2, 520, 1000), (3, 72, 250), (7, 8, 2048), (8, 5120, 12288),
         (15, 2048, 2040), (16, 640, 4096), (17, 1024, 1000), (31, 3000, 520 + 8),
         (32, 5120, 4096), (33, 136, 2048), (48, 1024, 256), (63, 4096, 1000), (64, 5120, 12288)]


@pytest.mark.parametrize("M,K,N", [c for c in CASES if si.nblocks(c[2]) % 8 == 0])
def test_skinny_parity(M, K, N):
    A = si.activations_bf16(M, K, seed=M + K)
    B = si.q4_weights(K, N, seed=N + 1)
    C = tiles(A, B, M, N, K)
    if M * N <= 64 * 4096:
        check_tiles(C, A, B, M, N, K, f"M={M} K={K} N={N}")
    else:
        # 24 seeded block columns, every row and every K
        nb = si.nblocks(N)
        cols = np.sort(si.rng(M, 5).choice(nb, size=24, replace=False))
        Bs = B.reshape(K, nb, 18)[:, cols].reshape(K, -1)
        got = to_host64(C).reshape(M, nb, 32)[:, cols].reshape(M, -1)
        Cb, Sb = oracle.matmul_bf16_tiles(A, Bs, M, 32 * len(cols), K)
        assert (np.abs(got - Cb) <= 1e-4 * Sb + 1e-6).all(), f"M={M} K={K} N={N}"


@pytest.mark.parametrize("M", [1, 5, 16, 24, 40, 64])
def test_skinny_one_hot_rows_give_bf16_tiles(M):
    """Row i of A = e_{k_i}: C row i is the bf16 tile row k_i exactly (one
    nonzero product per sum, the other slices add exact zeros)."""
    K, N = 3000, 1000
    B = si.q4_weights(K, N, seed=41 + M)
    ks = si.rng(41, M).choice(K, size=M, replace=False)
    A = np.zeros((M, K), np.float32)
    A[np.arange(M), ks] = 1.0
    C = tiles(si.f32_to_bf16_bits(A), B, M, N, K).cpu().numpy()
    Wb = oracle.dequant_bf16(B, K, N)
    assert np.array_equal(C, (Wb[ks].astype(np.uint32) << 16).view(np.float32))


def test_skinny_golden_tile_blocks():
    """Hand-rounded bf16 tile values (ties to even) come out of the few-row
    form's dequant, read back through one-hot rows."""
    import test_oracle_pins as pins
    recs = pins._golden_bf16_blocks()
    K, N, M = 64, 256, 64
    blocks = [blk for _, blk, _ in recs]
    B = np.frombuffer(b"".join(blocks[(k + b) % len(blocks)] for k in range(K) for b in range(8)),
                      np.uint8).reshape(K, 8 * 18)
    A = np.zeros((M, K), np.float32)
    A[np.arange(M), np.arange(M) % K] = 1.0
    C = tiles(si.f32_to_bf16_bits(A), B, M, N, K).cpu().numpy()
    for i in range(M):
        k = i % K
        for b in range(8):
            want = np.array(recs[(k + b) % len(recs)][2], np.float32)
            assert np.array_equal(C[i, 32 * b:32 * b + 32], want), (i, b)


@pytest.mark.parametrize("M", [2, 8, 40, 64])
def test_skinny_deterministic_bf16_output(M):
    K, N = 5120, 2048
    A = si.activations_bf16(M, K, seed=60 + M)
    B = si.q4_weights(K, N, seed=60)
    c1 = tiles(A, B, M, N, K)
    c2 = tiles(A, B, M, N, K)
    c16 = tiles(A, B, M, N, K, c_dtype=torch.bfloat16)
    assert torch.equal(c1, c2)
    assert torch.equal(c1.to(torch.bfloat16).view(torch.int16), c16.view(torch.int16))


def test_skinny_one_slice_per_tile():
    """More 256-column tiles than SMs: each CTA streams its tile's whole K
    and stores C directly (no partial tiles)."""
    M, K, N = 4, 1024, 256 * 160
    A = si.activations_bf16(M, K, seed=7)
    B = si.q4_weights(K, N, seed=7)
    C = tiles(A, B, M, N, K)
    nb = si.nblocks(N)
    cols = np.unique(np.concatenate([[0, nb - 1], si.rng(7, 1).choice(nb, 22, replace=False)]))
    Bs = B.reshape(K, nb, 18)[:, cols].reshape(K, -1)
    got = to_host64(C).reshape(M, nb, 32)[:, cols].reshape(M, -1)
    Cb, Sb = oracle.matmul_bf16_tiles(A, Bs, M, 32 * len(cols), K)
    assert (np.abs(got - Cb) <= 1e-4 * Sb + 1e-6).all()


@pytest.mark.parametrize("M", [2, 4, 8, 32, 64])
def test_skinny_through_matmul_ex(M):
    """q4_matmul_ex routes bf16 A with 4 <= M <= 32 and K >= 1024 here (M = 2
    to the exact GEMV, M = 64 to the split forms); the stated tolerance holds
    on the seeded data."""
    K, N = 5120, 12288
    A = si.activations_bf16(M, K, seed=70 + M)
    B = si.q4_weights(K, N, seed=70)
    C = torch.empty((M, N), dtype=torch.float32, device=device())
    q4.q4_matmul_ex(C, to_dev(A), to_dev(B), M, N, K)
    torch.cuda.synchronize()
    assert q4.q4_get_device_status() == q4.Q4_OK
    nb = si.nblocks(N)
    cols = np.sort(si.rng(M, 6).choice(nb, size=16, replace=False))
    Bs = B.reshape(K, nb, 18)[:, cols].reshape(K, -1)
    got = to_host64(C).reshape(M, nb, 32)[:, cols].reshape(M, -1)
    C64, S = oracle.matmul(A, Bs, M, 32 * len(cols), K)
    assert_within_matmul_tol(got, C64, S, f"q4_matmul_ex M={M}")
    if M >= 4:   # the tensor-core forms: A . bf16_rn(W)
        Cb, Sb = oracle.matmul_bf16_tiles(A, Bs, M, 32 * len(cols), K)
        assert (np.abs(got - Cb) <= 1e-4 * Sb + 1e-6).all()


@pytest.mark.parametrize("M", [4, 32])
def test_skinny_workspace_in_a_graph(M):
    """A zeroed caller workspace carries the slices' partial tiles and
    tickets, eagerly and in a captured graph; replays equal the eager call
    and leave the tickets at zero."""
    K, N = 4096, 8192
    nbytes = q4.q4_matmul_workspace_size(M, N, K)
    assert nbytes > 0
    ws = torch.zeros(nbytes, dtype=torch.uint8, device=device())
    A = si.activations_bf16(M, K, seed=80 + M)
    B = si.q4_weights(K, N, seed=80)
    dA, dB = to_dev(A), to_dev(B)
    s = torch.cuda.Stream()
    eager = torch.empty((M, N), dtype=torch.float32, device=device())
    with torch.cuda.stream(s):
        q4.q4_matmul_ex(eager, dA, dB, M, N, K, workspace=ws, stream=s)
    s.synchronize()
    cap = torch.empty_like(eager)
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        q4.q4_matmul_ex(cap, dA, dB, M, N, K, workspace=ws, stream=s)
    for _ in range(3):
        g.replay()
    torch.cuda.synchronize()
    assert q4.q4_get_device_status() == q4.Q4_OK
    assert torch.equal(cap, eager)
    assert not ws[:4 * ((N + 255) // 256)].cpu().numpy().any()
    nb = si.nblocks(N)
    cols = np.sort(si.rng(M, 8).choice(nb, size=16, replace=False))
    Bs = B.reshape(K, nb, 18)[:, cols].reshape(K, -1)
    got = to_host64(eager).reshape(M, nb, 32)[:, cols].reshape(M, -1)
    Cb, Sb = oracle.matmul_bf16_tiles(A, Bs, M, 32 * len(cols), K)
    assert (np.abs(got - Cb) <= 1e-4 * Sb + 1e-6).all()
