"""Seeded random shapes through q4_matmul_ex (both weight formats, both
activation types, both output types), each compared with the oracle element
by element at the stated tolerance, and the tensor-core GEMM
(q4_matmul_bf16_tiles) against its bf16-tile oracle.

The shapes are drawn so that the cases cross the launch-shape choices: one
or several rows of A (the GEMV's chunks of 1, 2 and 4 rows), ceil(N/32) a
multiple of 8 or not (tensor copies or the producer-warp copy), K slices with
and without a ragged last stage, and M from 8 up on the tensor cores.
"""

import numpy as np
import pytest

import oracle
import seeded_inputs as si
from gpu_util import assert_within_matmul_tol, device, to_dev, to_host64, torch

import quantized_weight_q4_gb300 as q4

pytestmark = pytest.mark.gpu


def draw_cases(n, seed, m_hi, q8_ok):
    g = si.rng(seed, 77)
    cases = []
    for i in range(n):
        M = int(g.integers(1, 5)) if g.random() < 0.5 else int(g.integers(5, m_hi + 1))
        K = int(g.integers(1, 3000))
        nb = int(g.integers(1, 80))
        if g.random() < 0.5:
            nb = 8 * max(1, nb // 8)          # tensor-copy friendly rows
        N = 32 * nb - int(g.integers(0, 32))
        adt = "bf16" if g.random() < 0.5 else "f32"
        cdt = torch.bfloat16 if g.random() < 0.25 else torch.float32
        fmt = "q8" if (q8_ok and g.random() < 0.3) else "q4"
        cases.append((i, M, K, N, adt, cdt, fmt))
    return cases


def check(i, M, K, N, adt, cdt, fmt):
    A = si.activations_bf16(M, K, seed=i) if adt == "bf16" else si.activations_f32(M, K, seed=i)
    q8 = fmt == "q8"
    B = (si.q8_weights if q8 else si.q4_weights)(K, N, seed=i + 1000)
    C = torch.empty((M, N), dtype=cdt, device=device())
    q4.q4_matmul_ex(C, to_dev(A), to_dev(B), M, N, K,
                    b_layout=q4.Q4_LAYOUT_Q8_0 if q8 else q4.Q4_LAYOUT_BLOCKS)
    torch.cuda.synchronize()
    assert q4.q4_get_device_status() == q4.Q4_OK
    C64, S = (oracle.q8_matmul if q8 else oracle.matmul)(A, B, M, N, K)
    what = f"case {i}: M={M} K={K} N={N} {adt} {cdt} {fmt}"
    got = to_host64(C)
    if cdt == torch.bfloat16:
        # the fp32 result rounded once more to bf16
        err = np.abs(got - C64)
        assert (err <= 1e-3 * S + 1e-6 + 2.0 ** -8 * np.abs(C64)).all(), what
    else:
        assert_within_matmul_tol(got, C64, S, what)


@pytest.mark.parametrize("case", draw_cases(40, seed=1, m_hi=64, q8_ok=True),
                         ids=lambda c: f"{c[0]}-M{c[1]}K{c[2]}N{c[3]}{c[4]}{c[6]}")
def test_random_gemv_shapes(case):
    check(*case)


def tensor_cases():
    out = []
    g = si.rng(2, 78)
    for i in range(12):
        M = int(g.choice([8, 9, 16, 33, 64, 100, 128, 129, 200, 256]))
        K = 8 * int(g.integers(1, 400))
        N = 256 * int(g.integers(1, 12))
        out.append((100 + i, M, K, N, "bf16", torch.float32, "q4"))
    return out


@pytest.mark.parametrize("case", tensor_cases(), ids=lambda c: f"{c[0]}-M{c[1]}K{c[2]}N{c[3]}")
def test_random_tensor_core_shapes(case):
    """bf16 A with M >= 8 and tensor-core shapes.  q4_matmul_ex (the GEMM from
    K = 1024 on, the exact GEMV below) within the stated tolerance; the GEMM
    itself (q4_matmul_bf16_tiles) within 1e-4 of A . bf16_rn(W) and within the
    bf16 rounding bound of A . W at any K."""
    i, M, K, N, _, _, _ = case
    A = si.activations_bf16(M, K, seed=i)
    B = si.q4_weights(K, N, seed=i + 1000)
    dA, dB = to_dev(A), to_dev(B)
    C = torch.empty((M, N), dtype=torch.float32, device=device())
    q4.q4_matmul_ex(C, dA, dB, M, N, K)
    torch.cuda.synchronize()
    assert q4.q4_get_device_status() == q4.Q4_OK
    C64, S = oracle.matmul(A, B, M, N, K)
    assert_within_matmul_tol(to_host64(C), C64, S, f"q4_matmul_ex M={M} K={K} N={N}")
    q4.q4_matmul_bf16_tiles(C, dA, dB, M, N, K)
    torch.cuda.synchronize()
    assert q4.q4_get_device_status() == q4.Q4_OK
    got = to_host64(C)
    Cb, Sb = oracle.matmul_bf16_tiles(A, B, M, N, K)
    assert (np.abs(got - Cb) <= 1e-4 * Sb + 1e-6).all(), f"tiles M={M} K={K} N={N}"
    assert (np.abs(got - C64) <= (2.0 ** -8 + 1e-4) * S + 1e-6).all(), f"tiles M={M} K={K} N={N}"
