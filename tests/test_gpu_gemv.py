"""GPU Q4_0 GEMV (M <= 64) against the fp64 oracle, element by element.

Tolerance: |gpu - oracle| <= 1e-3 * sum_k |a*w| + 1e-6 per output element.
Exact cases (one-hot A, padding, zeros, determinism) are compared bit for bit.
"""

import numpy as np
import pytest

import oracle
import seeded_inputs as si
from gpu_util import assert_within_matmul_tol, device, to_dev, to_host64, torch

import quantized_weight_q4_gb300 as q4

pytestmark = pytest.mark.gpu


def run(A, B, M, N, K, c_dtype=torch.float32, workspace=None):
    C = torch.empty((M, N), dtype=c_dtype, device=device())
    q4.q4_matmul_ex(C, to_dev(A), to_dev(B), M, N, K, workspace=workspace)
    torch.cuda.synchronize()
    return C


SHAPES = [
    (1, 1, 32), (1, 7, 40), (1, 64, 256), (1, 100, 1000), (1, 4096, 4096),
    (2, 333, 300), (2, 1000, 2048), (3, 64, 96), (4, 515, 800), (4, 1024, 4352),
    (5, 200, 520), (8, 300, 256), (17, 129, 1056), (64, 256, 512),
]


@pytest.mark.parametrize("M,K,N", SHAPES)
@pytest.mark.parametrize("adt", ["f32", "bf16"])
def test_gemv_parity(M, K, N, adt):
    A = si.activations_f32(M, K, seed=M * K) if adt == "f32" else si.activations_bf16(M, K, seed=M * K)
    B = si.q4_weights(K, N, seed=N)
    C = to_host64(run(A, B, M, N, K))
    C64, S = oracle.matmul(A, B, M, N, K)
    assert_within_matmul_tol(C, C64, S, f"M={M} K={K} N={N} {adt}")


@pytest.mark.parametrize("M,K,N", [(1, 100, 1000), (4, 515, 800), (2, 4096, 4096)])
def test_bf16_output_is_rounded_fp32(M, K, N):
    A = si.activations_bf16(M, K, seed=3)
    B = si.q4_weights(K, N, seed=3)
    C32 = run(A, B, M, N, K)
    C16 = run(A, B, M, N, K, c_dtype=torch.bfloat16)
    assert torch.equal(C32.to(torch.bfloat16).view(torch.int16), C16.view(torch.int16))


@pytest.mark.parametrize("K,N", [(9, 96), (300, 256), (1000, 4096)])
def test_one_hot_rows_are_exact(K, N):
    """A = e_k selects row k of W: exact in fp32 (only zeros are added)."""
    B = si.q4_weights(K, N, seed=11)
    W = oracle.dequant_f32(B, K, N)
    ks = sorted({0, K // 3, K - 1})
    A = np.zeros((len(ks), K), np.float32)
    for i, k in enumerate(ks):
        A[i, k] = 1.0
    for i, k in enumerate(ks):
        C = run(A[i:i + 1], B, 1, N, K).cpu().numpy()
        assert np.array_equal(C[0], W[k]), k
    C = run(A, B, len(ks), N, K).cpu().numpy()
    assert np.array_equal(C, W[ks])


@pytest.mark.parametrize("K,N", [(50, 40), (700, 1000), (64, 33)])
def test_padding_never_contributes(K, N):
    A = si.activations_f32(3, K, seed=5)
    B = si.q4_weights(K, N, seed=5)
    Br = si.randomise_padding(B, K, N, seed=5, stream=99)
    C = run(A, B, 3, N, K).cpu().numpy()
    Cr = run(A, Br, 3, N, K).cpu().numpy()
    assert np.array_equal(C, Cr)


def test_zero_inputs_give_zero():
    K, N = 500, 768
    B = si.q4_weights(K, N, seed=2)
    Z = B.reshape(K, -1, 18).copy()
    Z[:, :, 2:] = 0x88
    A = si.activations_f32(2, K, seed=2)
    assert not run(A, Z.reshape(K, -1), 2, N, K).any()
    assert not run(np.zeros((2, K), np.float32), B, 2, N, K).any()


def test_deterministic():
    M, K, N = 1, 4096, 11008
    A = si.activations_f32(M, K, seed=8)
    B = si.q4_weights(K, N, seed=8)
    c1 = run(A, B, M, N, K)
    c2 = run(A, B, M, N, K)
    assert torch.equal(c1, c2)


def test_single_gemv_4096():
    """One Q4_0 GEMV: M = 1, K = N = 4096, fp32 A, every output checked."""
    M, K, N = 1, 4096, 4096
    A = si.activations_f32(M, K, seed=0)
    B = si.q4_weights(K, N, seed=0)
    C = to_host64(run(A, B, M, N, K))
    C64, S = oracle.matmul(A, B, M, N, K)
    assert_within_matmul_tol(C, C64, S, "4096x4096")


@pytest.mark.parametrize("M", [1, 2, 4, 8, 16, 32, 64])
def test_batched_decode_5120x12288(M):
    """K = 5120, N = 12288, bf16 A with M rows: every row, a sample of 24
    block columns (768 output columns) computed by the oracle."""
    K, N = 5120, 12288
    A = si.activations_bf16(M, K, seed=M)
    B = si.q4_weights(K, N, seed=0)
    C = to_host64(run(A, B, M, N, K))
    nb = si.nblocks(N)
    cols = np.sort(si.rng(M, 3).choice(nb, size=24, replace=False))
    cols[-1] = nb - 1
    Bs = B.reshape(K, nb, 18)[:, cols, :].reshape(K, -1)
    C64, S = oracle.matmul(A, Bs, M, 32 * len(cols), K)
    got = C.reshape(M, nb, 32)[:, cols, :].reshape(M, -1)
    assert_within_matmul_tol(got, C64, S, f"M={M}")


def test_gemv_needs_no_workspace():
    """The GEMV combines its split-K partial sums on chip: a caller-provided
    workspace is ignored (q4_matmul_workspace_size reports what the
    tensor-core forms of the same shape may use)."""
    M, K, N = 1, 4096, 4096
    A = si.activations_f32(M, K, seed=1)
    B = si.q4_weights(K, N, seed=1)
    ws = torch.zeros(256, dtype=torch.uint8, device=device())
    c1 = run(A, B, M, N, K, workspace=ws)
    c2 = run(A, B, M, N, K)
    assert torch.equal(c1, c2)


def test_moe_workspace_too_small_rejected():
    T, topk, E, H, I = 2, 2, 4, 256, 64
    need = q4.q4_moe_workspace_size(T, topk, E, H, I)
    assert need > 0
    out = torch.empty((T, H), dtype=torch.float32, device=device())
    x = to_dev(si.activations_bf16(T, H, 1))
    W = to_dev(np.zeros((E, H, 2 * 18), np.uint8))
    Wd = to_dev(np.zeros((E, I, 8 * 18), np.uint8))
    idx = to_dev(np.zeros((T, topk), np.int32))
    w = to_dev(np.zeros((T, topk), np.float32))
    small = torch.zeros(need // 2, dtype=torch.uint8, device=device())
    with pytest.raises(q4.Q4Error) as e:
        q4.q4_moe_experts_ex(out, x, W, W, Wd, idx, w, T, topk, E, H, I, workspace=small)
    assert e.value.status == q4.Q4_ERR_WORKSPACE


def test_misaligned_pointer_rejected():
    K, N = 64, 256
    B = to_dev(si.q4_weights(K, N, seed=1))
    A = torch.zeros(K + 4, dtype=torch.float32, device=device())
    C = torch.empty((1, N), dtype=torch.float32, device=device())
    with pytest.raises(q4.Q4Error) as e:
        q4.q4_matmul_ex(C, A[1:K + 1], B, 1, N, K)
    assert e.value.status == q4.Q4_ERR_ALIGN


def test_decode_sweep_graph():
    """The 7B-like decode sweep (32 layers x 7 GEMVs, M = 1, fp32 A, ~3.6 GB of
    weights) captured in one CUDA graph, as the benchmark runs it; outputs are
    checked on 2 sampled block columns of every one of the 224 GEMVs."""
    from quantized_weight_q4_gb300.graph import MatmulSequence
    shapes = si.sweep_shapes()
    calls, host = [], []
    for i, (K, N) in enumerate(shapes):
        B = si.q4_weights(K, N, seed=0, stream=100 + i)
        A = si.activations_f32(1, K, seed=0, stream=10000 + i)
        nb = si.nblocks(N)
        cols = si.rng(i, 1).choice(nb, size=2, replace=False)
        host.append((A, B.reshape(K, nb, 18)[:, cols, :].reshape(K, -1).copy(), cols))
        C = torch.empty((1, N), dtype=torch.float32, device=device())
        calls.append((C, to_dev(A), to_dev(B), 1, N, K))
        del B
    seq = MatmulSequence(calls).capture()
    for C, *_ in calls:
        C.zero_()
    seq.replay()
    torch.cuda.synchronize()
    for (C, _, _, _, N, K), (A, Bs, cols) in zip(calls, host):
        got = to_host64(C).reshape(1, -1, 32)[:, cols, :].reshape(1, -1)
        C64, S = oracle.matmul(A, Bs, 1, 64, K)
        assert_within_matmul_tol(got, C64, S, f"K={K} N={N}")
