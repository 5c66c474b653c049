"""Pins of the oracle's Q8_0 functions (a second format behind the same
interface; the pages name Q8_0 but print no layout, so the reading is the
oracle's: fp16 d, then 32 two's-complement int8 codes, value = code * d,
blocks along the output columns as for Q4_0).

Each pin checks the oracle against something other than itself: hand-written
values, an exact re-encoding of pinned Q4_0 matrices, exact rational sums,
one-hot selection, padding invariance and linearity.
"""

import math
import os
from fractions import Fraction

import numpy as np
import pytest

import seeded_inputs as si

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "q8_0_blocks.txt")


def _golden():
    recs = []
    with open(GOLDEN) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            name, d, codes, vals = [p.strip() for p in line.split("|")]
            dbits = int(d, 16)
            cb = bytes(int(x, 16) for x in codes.split())
            assert len(cb) == 32
            v = [(-0.0 if t == "-0" else float(t)) for t in vals.split()]
            assert len(v) == 32
            recs.append((name, bytes([dbits & 0xFF, dbits >> 8]) + cb, v))
    return recs


def test_hand_written_blocks():
    import oracle
    recs = _golden()
    assert len(recs) >= 6
    for name, blk, vals in recs:
        W = oracle.q8_dequant_f32(np.frombuffer(blk, np.uint8).reshape(1, 34), 1, 32)
        for l in range(32):
            got, want = float(W[0, l]), vals[l]
            assert got == want and math.copysign(1, got) == math.copysign(1, want), (name, l)


def _q4_as_q8(B4, K, N):
    """Re-encodes Q4_0 blocks as Q8_0 blocks with the same scale and code q - 8
    (exact: -8..7 fits int8)."""
    nb = si.nblocks(N)
    b4 = B4.reshape(K, nb, 18)
    out = np.empty((K, nb, 34), np.uint8)
    out[:, :, :2] = b4[:, :, :2]
    qs = b4[:, :, 2:]
    codes = np.empty((K, nb, 32), np.int16)
    codes[:, :, 0::2] = qs & 0x0F
    codes[:, :, 1::2] = qs >> 4
    out[:, :, 2:] = ((codes - 8) & 0xFF).astype(np.uint8)
    return out.reshape(K, nb * 34)


@pytest.mark.parametrize("M,K,N", [(1, 7, 40), (2, 64, 96), (3, 100, 300)])
def test_equals_pinned_q4_on_reencoded_weights(M, K, N):
    """A Q4_0 matrix re-encoded as Q8_0 (same d, code q - 8) gives the same
    weights and, summed in the same order, the same fp64 products."""
    import oracle
    B4 = si.q4_weights(K, N, seed=M + K)
    B8 = _q4_as_q8(B4, K, N)
    assert np.array_equal(oracle.q8_dequant_f32(B8, K, N), oracle.dequant_f32(B4, K, N))
    A = si.activations_f32(M, K, seed=N)
    C8, S8 = oracle.q8_matmul(A, B8, M, N, K)
    C4, S4 = oracle.matmul(A, B4, M, N, K)
    assert np.array_equal(C8, C4) and np.array_equal(S8, S4)


def test_layout_one_hot():
    """A = e_k selects row k; a single non-zero block lands in its 32 columns."""
    import oracle
    K, N = 9, 100
    B = si.q8_weights(K, N, seed=4)
    W = oracle.q8_dequant_f32(B, K, N)
    for k in (0, 4, K - 1):
        A = np.zeros((1, K), np.float32)
        A[0, k] = 1.0
        C, _ = oracle.q8_matmul(A, B, 1, N, K)
        assert np.array_equal(C[0], W[k].astype(np.float64))
    Z = np.zeros_like(B).reshape(K, -1, 34)
    Z[5, 2, :2] = np.array([0x00, 0x3C], np.uint8)         # d = 1.0 in block (5, 2)
    Z[5, 2, 2:] = np.arange(32, dtype=np.uint8)            # codes 0..31
    Wz = oracle.q8_dequant_f32(Z.reshape(K, -1), K, N)
    nz = np.argwhere(Wz != 0)
    assert set(map(tuple, nz)) == {(5, j) for j in range(65, 96)}   # code 0 at column 64
    assert Wz[5, 64] == 0 and Wz[5, 95] == 31


def _exact(A, W):
    M, K = A.shape
    N = W.shape[1]
    out = [[Fraction(0)] * N for _ in range(M)]
    for i in range(M):
        for k in range(K):
            a = Fraction(float(A[i, k]))
            for j in range(N):
                out[i][j] += a * Fraction(float(W[k, j]))
    return out


@pytest.mark.parametrize("M,K,N", [(1, 1, 32), (2, 5, 40), (1, 33, 64)])
def test_exact_rational(M, K, N):
    import oracle
    B = si.q8_weights(K, N, seed=K + 1)
    A = si.activations_f32(M, K, seed=K + 2)
    W = oracle.q8_dequant_f32(B, K, N)
    C, S = oracle.q8_matmul(A, B, M, N, K)
    ex = _exact(A, W)
    for i in range(M):
        for j in range(N):
            err = abs(Fraction(C[i, j]) - ex[i][j])
            assert err <= Fraction(K * 2.0 ** -52) * Fraction(S[i, j]) + Fraction(1, 2 ** 1070)
            assert abs(C[i, j]) <= S[i, j]


def test_padding_and_linearity():
    import oracle
    K, N = 20, 70
    B = si.q8_weights(K, N, seed=3)
    Br = B.copy().reshape(K, -1, 34)
    Br[:, -1, 2 + (N - 64):] = si.rng(3, 9).integers(0, 256, size=(K, 32 - (N - 64)), dtype=np.uint8)
    A1 = si.activations_f32(2, K, seed=1)
    A2 = si.activations_f32(2, K, seed=2)
    C, _ = oracle.q8_matmul(A1, B, 2, N, K)
    Cr, _ = oracle.q8_matmul(A1, Br.reshape(K, -1), 2, N, K)
    assert np.array_equal(C, Cr)
    C2, _ = oracle.q8_matmul(A2, B, 2, N, K)
    C12, S12 = oracle.q8_matmul((A1.astype(np.float64) + A2).astype(np.float32), B, 2, N, K)
    # A1 + A2 rounds once in fp32: compare within that rounding and the sums' bound
    assert np.all(np.abs(C12 - (C + C2)) <= 2.0 ** -23 * S12 * 2 + 1e-30)
