"""Pins of the fp64 CPU oracle against what the pages and mathematics fix.

Nothing here calls the CUDA path.  Each test ties an oracle function to
something other than itself: a library conversion over every code, blocks
whose values were worked out by hand from the block definition (C++ DeepSeek
engine page, §2.2), exact rational sums, one-hot / zero / scaling / padding
invariants, and closed forms of SiLU for the routed-expert chain
(KTransformers DeepSeek-V2 page, «优化三»).
"""

import math
import os
from fractions import Fraction

import numpy as np
import pytest

import seeded_inputs as si

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "q4_0_blocks.txt")


def _golden_blocks():
    recs = []
    with open(GOLDEN) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            name, d, qs, vals = [p.strip() for p in line.split("|")]
            dbits = int(d, 16)
            qsb = bytes(int(x, 16) for x in qs.split())
            assert len(qsb) == 16
            blk = bytes([dbits & 0xFF, dbits >> 8]) + qsb
            special = {"inf": math.inf, "-inf": -math.inf, "nan": math.nan,
                       "-0": -0.0, "0": 0.0}
            v = [special[t] if t in special else float(t) for t in vals.split()]
            assert len(v) == 32
            recs.append((name, blk, v))
    return recs


def _same(a: float, b: float) -> bool:
    """Equal including the sign of zero; NaN matches NaN."""
    if math.isnan(a) or math.isnan(b):
        return math.isnan(a) and math.isnan(b)
    return a == b and math.copysign(1.0, a) == math.copysign(1.0, b)


# ---------------------------------------------------------------- formats

def test_fp16_decode_all_codes(oracle_lib):
    """The oracle's binary16 decode equals numpy's for all 65536 codes."""
    codes = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    ref = codes.view(np.float16).astype(np.float64)
    for c in range(65536):
        got = oracle_lib.fp16_to_f64(c)
        assert _same(got, float(ref[c])), hex(c)


def test_bf16_decode_all_codes(oracle_lib):
    """bf16 decode equals the fp32 whose upper half is the code, for all codes."""
    codes = np.arange(65536, dtype=np.uint32)
    with np.errstate(invalid="ignore"):
        ref = (codes << 16).astype(np.uint32).view(np.float32).astype(np.float64)
    for c in range(65536):
        assert _same(oracle_lib.bf16_to_f64(c), float(ref[c])), hex(c)


def test_bf16_encode_matches_torch(oracle_lib):
    """fp64 -> bf16 round-to-nearest-even equals torch's fp32 -> bf16 cast,
    on random values and on exact ties (inputs exactly representable in fp32)."""
    torch = pytest.importorskip("torch")
    g = si.rng(7, 0)
    with np.errstate(over="ignore"):
        x = np.concatenate([
            g.standard_normal(20000).astype(np.float32),
            (g.standard_normal(2000) * 1e-38).astype(np.float32),   # bf16 subnormals
            (g.standard_normal(2000) * 3e38).astype(np.float32),    # overflow to inf
        ])
    # ties: bf16 value + half an ulp, both parities
    base = (g.integers(0, 0x7F00, 4000).astype(np.uint32) << 16)
    ties = (base | 0x8000).view(np.float32)
    x = np.concatenate([x, ties, -ties, np.array([0.0, -0.0, np.inf, -np.inf], np.float32)])
    ref = torch.from_numpy(x).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    for xi, r in zip(x, ref):
        assert oracle_lib.f64_to_bf16(float(xi)) == int(r), (float(xi), hex(int(r)))


# ---------------------------------------------------------------- dequant

def test_dequant_hand_built_blocks(oracle_lib):
    """Every hand-built block dequantises to the hand-derived values."""
    for name, blk, vals in _golden_blocks():
        W = oracle_lib.dequant_f32(np.frombuffer(blk, np.uint8), 1, 32)
        for l in range(32):
            assert _same(float(W[0, l]), vals[l]), (name, l, W[0, l], vals[l])


def test_dequant_all_nibbles_both_positions(oracle_lib):
    """All 16 codes in both nibble positions, for several scales: value = (q-8)*d."""
    for dbits in (0x3C00, 0xBC00, 0x3800, 0x0400, 0x03FF, 0x5640):
        d = float(np.array([dbits], np.uint16).view(np.float16)[0])
        for q in range(16):
            lo = bytes([dbits & 0xFF, dbits >> 8]) + bytes([0x80 | q] * 16)       # lo = q, hi = 8
            hi = bytes([dbits & 0xFF, dbits >> 8]) + bytes([(q << 4) | 8] * 16)   # lo = 8, hi = q
            Wlo = oracle_lib.dequant_f32(np.frombuffer(lo, np.uint8), 1, 32)[0]
            Whi = oracle_lib.dequant_f32(np.frombuffer(hi, np.uint8), 1, 32)[0]
            for l in range(32):
                even = (l % 2 == 0)
                exp_lo = (q - 8) * d if even else 0.0 * d
                exp_hi = 0.0 * d if even else (q - 8) * d
                assert _same(float(Wlo[l]), float(np.float32(exp_lo))), (dbits, q, l)
                assert _same(float(Whi[l]), float(np.float32(exp_hi))), (dbits, q, l)


def test_dequant_bf16_is_rounded_f32(oracle_lib):
    """The bf16 tile value is the fp32 value rounded by torch's cast."""
    torch = pytest.importorskip("torch")
    K, N = 16, 96
    B = si.q4_weights(K, N, seed=3, d_lo=0.001, d_hi=40.0)
    W32 = oracle_lib.dequant_f32(B, K, N)
    W16 = oracle_lib.dequant_bf16(B, K, N)
    ref = torch.from_numpy(W32).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(W16, ref)


# ---------------------------------------------------------------- matmul

def _hand_matrix(K, N, k0, b0, qs_pattern, dbits=0x3C00):
    """K x N blocks with every code 8 (value 0) except block (k0, b0)."""
    nb = si.nblocks(N)
    B = np.zeros((K, nb, 18), np.uint8)
    B[:, :, 2:] = 0x88
    B[:, :, 0] = dbits & 0xFF
    B[:, :, 1] = dbits >> 8
    B[k0, b0, 2:] = np.frombuffer(bytes(qs_pattern), np.uint8)
    return B.reshape(K, nb * 18)


def test_layout_one_hot():
    """Only block (k0, b0) is non-zero: a one-hot A on row k0 reads the ramp
    into columns 32*b0 .. 32*b0+31 and nowhere else; other rows give zero."""
    import oracle
    K, N, k0, b0 = 5, 96, 3, 1
    ramp = [0x10, 0x32, 0x54, 0x76, 0x98, 0xBA, 0xDC, 0xFE] * 2
    B = _hand_matrix(K, N, k0, b0, ramp)
    for k in range(K):
        A = np.zeros((1, K), np.float32)
        A[0, k] = 1.0
        C, _ = oracle.matmul(A, B, 1, N, K)
        exp = np.zeros(N)
        if k == k0:
            exp[32 * b0:32 * b0 + 32] = [(l % 16) - 8 for l in range(32)]
        assert np.array_equal(C[0], exp), k


def test_zero_cases():
    import oracle
    K, N = 7, 64
    A = si.activations_f32(2, K, seed=1)
    B = si.q4_weights(K, N, seed=1)
    # all codes 8
    Z = B.reshape(K, -1, 18).copy()
    Z[:, :, 2:] = 0x88
    C, S = oracle.matmul(A, Z.reshape(K, -1), 2, N, K)
    assert np.all(C == 0) and np.all(S == 0)
    # d = +0 and d = -0
    for lo, hi in ((0, 0), (0, 0x80)):
        Z = B.reshape(K, -1, 18).copy()
        Z[:, :, 0], Z[:, :, 1] = lo, hi
        C, _ = oracle.matmul(A, Z.reshape(K, -1), 2, N, K)
        assert np.all(C == 0)
    # A = 0
    C, _ = oracle.matmul(np.zeros((2, K), np.float32), B, 2, N, K)
    assert np.all(C == 0)


def _exact_product(A, W):
    """Exact rational A . W from the fp32 values (no rounding anywhere)."""
    M, K = A.shape
    N = W.shape[1]
    out = [[Fraction(0)] * N for _ in range(M)]
    for i in range(M):
        for k in range(K):
            a = Fraction(float(A[i, k]))
            if a == 0:
                continue
            for j in range(N):
                out[i][j] += a * Fraction(float(W[k, j]))
    return out


@pytest.mark.parametrize("M,K,N", [(1, 1, 32), (2, 3, 64), (3, 17, 40), (1, 64, 96)])
def test_matmul_exact_rational(M, K, N):
    """C64 is within the fp64 summation bound of the exact rational sum, and
    S bounds |C|; on small-integer data every sum is exact."""
    import oracle
    A = si.activations_f32(M, K, seed=K)
    B = si.q4_weights(K, N, seed=K)
    W = oracle.dequant_f32(B, K, N)
    C, S = oracle.matmul(A, B, M, N, K)
    ex = _exact_product(A, W)
    for i in range(M):
        for j in range(N):
            err = abs(Fraction(C[i, j]) - ex[i][j])
            assert err <= Fraction(K * 2.0 ** -52) * Fraction(S[i, j]) + Fraction(1, 2 ** 1070)
            assert abs(C[i, j]) <= S[i, j]
    # integer activations and unit scales: everything is exact
    Ai = np.asarray(si.rng(K, 9).integers(-3, 4, size=(M, K)), np.float32)
    Bi = B.reshape(K, -1, 18).copy()
    Bi[:, :, 0], Bi[:, :, 1] = 0x00, 0x3C
    Bi = Bi.reshape(K, -1)
    Ci, _ = oracle.matmul(Ai, Bi, M, N, K)
    exi = _exact_product(Ai, oracle.dequant_f32(Bi, K, N))
    for i in range(M):
        for j in range(N):
            assert Fraction(Ci[i, j]) == exi[i][j]


def test_fused_equals_textbook():
    """The fused loop (engine page §3.4) and dequantise-then-triple-loop
    (§3.1) agree within the fp64 summation bound, for fp32 and bf16 A."""
    import oracle
    for dt in ("f32", "bf16"):
        M, K, N = 3, 200, 160
        A = si.activations_f32(M, K, 4) if dt == "f32" else si.activations_bf16(M, K, 4)
        B = si.q4_weights(K, N, seed=4)
        C, S = oracle.matmul(A, B, M, N, K)
        Cn = oracle.matmul_naive(A, B, M, N, K)
        assert np.all(np.abs(C - Cn) <= 2 * K * 2.0 ** -53 * S)


def test_scaling_is_exact():
    """Doubling every scale d (exact in fp16) or every activation doubles C exactly."""
    import oracle
    M, K, N = 2, 50, 96
    A = si.activations_f32(M, K, 5)
    B = si.q4_weights(K, N, seed=5)
    C, _ = oracle.matmul(A, B, M, N, K)
    d = B.reshape(K, -1, 18)[:, :, 0:2].copy().view(np.float16)
    B2 = B.reshape(K, -1, 18).copy()
    B2[:, :, 0:2] = (d * np.float16(2)).view(np.uint8)
    C2, _ = oracle.matmul(A, B2.reshape(K, -1), M, N, K)
    assert np.array_equal(C2, 2 * C)
    C3, _ = oracle.matmul(2 * A, B, M, N, K)
    assert np.array_equal(C3, 2 * C)


def test_padding_never_contributes():
    """Random codes in padding nibbles leave every real output bit-identical
    (engine page §2.3: columns padded to a multiple of 32)."""
    import oracle
    for N in (1, 33, 40, 95):
        K = 9
        A = si.activations_f32(2, K, 6)
        B = si.q4_weights(K, N, seed=6)
        Br = si.randomise_padding(B, K, N, seed=6, stream=77)
        assert not np.array_equal(B, Br) or N % 32 == 0
        C, S = oracle.matmul(A, B, 2, N, K)
        Cr, Sr = oracle.matmul(A, Br, 2, N, K)
        assert np.array_equal(C, Cr) and np.array_equal(S, Sr)


def test_generator_padding_is_zero_code():
    """Padding columns hold the zero code q = 8 (reading of 'padding set to zero')."""
    K, N = 3, 40
    B = si.q4_weights(K, N, seed=1).reshape(K, 2, 18)
    last = B[:, 1, 2:]
    for l in range(N - 32, 32):
        q = (last[:, l // 2] >> (4 * (l % 2))) & 15
        assert np.all(q == 8)


# ---------------------------------------------------------------- experts

def _expert_closed_form(E, gcodes, ucodes):
    """H = I = 32 experts whose chain is computable by hand.

    W_gate[e] row 0 holds codes gcodes[e] with d = 1 (other rows zero code),
    W_up[e] row 0 holds codes ucodes[e], W_down[e] is the identity (row i has
    code 9 in column i, code 8 elsewhere, d = 1).  With x = e_0 this gives
    g = q_gate - 8, u = q_up - 8, y = h.
    """
    H = I = 32

    def mat(codes_row0):
        B = np.zeros((H, 1, 18), np.uint8)
        B[:, :, 0], B[:, :, 1] = 0x00, 0x3C
        B[:, :, 2:] = 0x88
        for l, q in enumerate(codes_row0):
            b = 2 + l // 2
            if l % 2 == 0:
                B[0, 0, b] = (B[0, 0, b] & 0xF0) | q
            else:
                B[0, 0, b] = (B[0, 0, b] & 0x0F) | (q << 4)
        return B.reshape(H, 18)

    ident = np.zeros((I, 1, 18), np.uint8)
    ident[:, :, 0], ident[:, :, 1] = 0x00, 0x3C
    ident[:, :, 2:] = 0x88
    for i in range(I):
        b = 2 + i // 2
        ident[i, 0, b] = (ident[i, 0, b] & (0x0F if i % 2 else 0xF0)) | (9 << (4 * (i % 2)))
    Wg = np.stack([mat(gcodes[e]) for e in range(E)])
    Wu = np.stack([mat(ucodes[e]) for e in range(E)])
    Wd = np.stack([ident.reshape(I, 18)] * E)
    return Wg, Wu, Wd


def test_moe_closed_form():
    """out = sum_k w_k * SiLU(g_k) * u_k with g, u known integers; SiLU from
    its definition g / (1 + e^-g), evaluated with Python's math module."""
    import oracle
    E, H, I, T, topk = 3, 32, 32, 1, 2
    gcodes = [[(l % 16) for l in range(32)], [8] * 32, [(15 - l % 16) for l in range(32)]]
    ucodes = [[9 + (l % 3) for l in range(32)], [(l % 16) for l in range(32)], [10] * 32]
    Wg, Wu, Wd = _expert_closed_form(E, gcodes, ucodes)
    x = np.zeros((T, H), np.float32)
    x[0, 0] = 1.0
    idx = np.array([[2, 0]], np.int32)
    w = np.array([[0.25, 0.75]], np.float32)
    out, tol, (g, u, h) = oracle.moe(x, Wg, Wu, Wd, idx, w, T, topk, E, H, I, stages=True)
    for j in range(H):
        exp = 0.0
        for k, e in enumerate(idx[0]):
            gv = gcodes[e][j] - 8
            uv = ucodes[e][j] - 8
            exp += float(w[0, k]) * (gv / (1.0 + math.exp(-gv))) * uv
        assert abs(out[0, j] - exp) <= 1e-15 * (1 + abs(exp)), j
        assert tol[0, j] >= 1e-6
    # expert 1 has g = 0 everywhere: SiLU(0) = 0, so routing only to it gives 0
    out1, _, _ = oracle.moe(x, Wg, Wu, Wd, np.array([[1, 1]], np.int32), w, T, topk, E, H, I)
    assert np.all(out1 == 0)


def test_moe_closed_form_two_tokens():
    """Each token's experts read that token's row of x: token 0 is e_0, token 1
    is 2 * e_0 (so its g and u double), with different routings."""
    import oracle
    E, H, I, T, topk = 3, 32, 32, 2, 2
    gcodes = [[(l % 16) for l in range(32)], [8] * 32, [(15 - l % 16) for l in range(32)]]
    ucodes = [[9 + (l % 3) for l in range(32)], [(l % 16) for l in range(32)], [10] * 32]
    Wg, Wu, Wd = _expert_closed_form(E, gcodes, ucodes)
    x = np.zeros((T, H), np.float32)
    x[0, 0] = 1.0
    x[1, 0] = 2.0
    idx = np.array([[2, 0], [0, 2]], np.int32)
    w = np.array([[0.25, 0.75], [0.5, 0.5]], np.float32)
    out, _, _ = oracle.moe(x, Wg, Wu, Wd, idx, w, T, topk, E, H, I, stages=True)
    for t in range(T):
        s = float(x[t, 0])
        for j in range(H):
            exp = 0.0
            for k, e in enumerate(idx[t]):
                gv = s * (gcodes[e][j] - 8)
                uv = s * (ucodes[e][j] - 8)
                exp += float(w[t, k]) * (gv / (1.0 + math.exp(-gv))) * uv
            assert abs(out[t, j] - exp) <= 1e-15 * (1 + abs(exp)), (t, j)


def test_silu_closed_forms(oracle_lib):
    assert oracle_lib.silu(0.0) == 0.0
    assert abs(oracle_lib.silu(1.0) - 1.0 / (1.0 + math.exp(-1.0))) < 1e-16
    assert oracle_lib.silu(50.0) == pytest.approx(50.0, rel=1e-20)
    assert abs(oracle_lib.silu(-50.0)) < 1e-19
    # odd-part identity SiLU(x) - SiLU(-x) = x
    for xv in (0.3, 1.7, 4.2):
        assert abs(oracle_lib.silu(xv) - oracle_lib.silu(-xv) - xv) < 1e-15


def _small_moe(T=3, E=5, H=64, I=96, topk=2, seed=11):
    Wg = np.stack([si.q4_weights(H, I, seed, 10 + e) for e in range(E)])
    Wu = np.stack([si.q4_weights(H, I, seed, 20 + e) for e in range(E)])
    Wd = np.stack([si.q4_weights(I, H, seed, 30 + e) for e in range(E)])
    x = si.activations_bf16(T, H, seed)
    idx, w = si.routing(T, E, topk, seed)
    return x, Wg, Wu, Wd, idx, w, T, topk, E, H, I


def test_moe_invalid_slots_and_linearity():
    import oracle
    x, Wg, Wu, Wd, idx, w, T, topk, E, H, I = _small_moe()
    out, _, _ = oracle.moe(x, Wg, Wu, Wd, idx, w, T, topk, E, H, I)
    # an out-of-range index contributes nothing
    bad = idx.copy()
    bad[:, 1] = E
    wb = w.copy()
    out_bad, _, _ = oracle.moe(x, Wg, Wu, Wd, bad, wb, T, topk, E, H, I)
    only0 = w.copy()
    only0[:, 1] = 0.0
    out0, _, _ = oracle.moe(x, Wg, Wu, Wd, idx, only0, T, topk, E, H, I)
    assert np.array_equal(out_bad, out0)
    bad[:, 1] = -1
    out_neg, _, _ = oracle.moe(x, Wg, Wu, Wd, bad, wb, T, topk, E, H, I)
    assert np.array_equal(out_neg, out0)
    # linear in the routing weights
    only1 = w.copy()
    only1[:, 0] = 0.0
    out1, _, _ = oracle.moe(x, Wg, Wu, Wd, idx, only1, T, topk, E, H, I)
    assert np.allclose(out0 + out1, out, rtol=0, atol=1e-12 * (1 + np.abs(out).max()))


def test_moe_expert_relabel_invariance():
    """Renaming experts (permuting the weight stacks and the indices together)
    leaves the output bit-identical."""
    import oracle
    x, Wg, Wu, Wd, idx, w, T, topk, E, H, I = _small_moe()
    out, tol, _ = oracle.moe(x, Wg, Wu, Wd, idx, w, T, topk, E, H, I)
    perm = np.array([3, 0, 4, 1, 2])           # new id of old expert e is perm[e]
    inv = np.argsort(perm)
    out2, tol2, _ = oracle.moe(x, Wg[inv], Wu[inv], Wd[inv], perm[idx].astype(np.int32), w,
                               T, topk, E, H, I)
    assert np.array_equal(out, out2) and np.array_equal(tol, tol2)


def test_moe_single_expert_is_matmul_chain():
    """With one slot of weight 1, out equals down(SiLU(gate x) * up x) built
    from the oracle's single-matmul pieces (stage values agree too)."""
    import oracle
    x, Wg, Wu, Wd, idx, w, T, topk, E, H, I = _small_moe(T=1, topk=1)
    w = np.ones_like(w)
    out, _, (g, u, h) = oracle.moe(x, Wg, Wu, Wd, idx, w, T, topk, E, H, I, stages=True)
    e = int(idx[0, 0])
    g2, _ = oracle.matmul(x, Wg[e], 1, I, H)
    u2, _ = oracle.matmul(x, Wu[e], 1, I, H)
    assert np.array_equal(g[0], g2[0]) and np.array_equal(u[0], u2[0])
    hv = np.array([oracle.silu(float(v)) for v in g2[0]]) * u2[0]
    assert np.allclose(h[0], hv, rtol=1e-15, atol=0)


# ---------------------------------------------------------------- bf16 tiles

GOLDEN_BF16 = os.path.join(os.path.dirname(__file__), "golden", "q4_0_bf16_tiles.txt")


def _golden_bf16_blocks():
    recs = []
    with open(GOLDEN_BF16) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            name, d, qs, vals = [p.strip() for p in line.split("|")]
            dbits = int(d, 16)
            blk = bytes([dbits & 0xFF, dbits >> 8]) + bytes(int(x, 16) for x in qs.split())
            v = [float(t) for t in vals.split()]
            assert len(blk) == 18 and len(v) == 32
            recs.append((name, blk, v))
    return recs


def test_bf16_tiles_hand_rounded():
    """One-hot rows of A select the bf16 tile values of hand-built blocks
    (rounded by hand, ties to even, in the fixture)."""
    import oracle
    recs = _golden_bf16_blocks()
    K, N = len(recs), 32
    B = np.frombuffer(b"".join(blk for _, blk, _ in recs), np.uint8).reshape(K, 18)
    A = si.f32_to_bf16_bits(np.eye(K, dtype=np.float32))
    C, S = oracle.matmul_bf16_tiles(A, B, K, N, K)
    for k, (name, _, vals) in enumerate(recs):
        assert np.array_equal(C[k], np.array(vals)), name
        assert np.array_equal(S[k], np.abs(np.array(vals))), name


def test_bf16_tiles_equal_exact_product_when_representable():
    """With power-of-two scales every weight (q-8)*d has at most 4 significant
    bits, so bf16 rounding changes nothing: the bf16-tile product equals the
    exact fused product up to fp64 summation order."""
    import oracle
    M, K, N = 5, 300, 96
    B = si.q4_weights(K, N, seed=21).reshape(K, -1, 18).copy()
    e = si.rng(21, 5).integers(-12, 2, size=B.shape[:2])
    d16 = np.ldexp(1.0, e).astype(np.float16).view(np.uint16)
    B[:, :, 0] = (d16 & 0xFF).astype(np.uint8)
    B[:, :, 1] = (d16 >> 8).astype(np.uint8)
    B = B.reshape(K, -1)
    A = si.activations_bf16(M, K, seed=21)
    Cb, Sb = oracle.matmul_bf16_tiles(A, B, M, N, K)
    C, S = oracle.matmul(A, B, M, N, K)
    assert np.all(np.abs(Cb - C) <= 1e-13 * S)
    assert np.allclose(Sb, S, rtol=1e-13, atol=0)


def test_bf16_tiles_within_rounding_bound():
    """bf16 carries 8 significant bits, so rounding to nearest moves a value by
    at most half its ulp, 2^-8 relative.  Every tile weight is within that of
    the exact one (and some weight is more than 2^-9 away: the bound is not
    loose by a factor of two), hence |A.bf16(W) - A.W| <= 2^-8 * sum_k |a*w|;
    with fp16 scales of 11 significant bits the rounding is not a no-op."""
    import oracle
    M, K, N = 4, 257, 160
    B = si.q4_weights(K, N, seed=22)
    W = oracle.dequant_f32(B, K, N).astype(np.float64)
    Wb = (oracle.dequant_bf16(B, K, N).astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    rel = np.abs(Wb - W) / np.maximum(np.abs(W), 1e-300)
    assert np.all(rel <= 2.0 ** -8)
    assert rel.max() > 2.0 ** -9
    A = si.activations_bf16(M, K, seed=22)
    Cb, _ = oracle.matmul_bf16_tiles(A, B, M, N, K)
    C, S = oracle.matmul(A, B, M, N, K)
    err = np.abs(Cb - C)
    assert np.all(err <= 2.0 ** -8 * S + 1e-300)
    assert err.max() > 0


# ---------------------------------------------------------------- router

def _softmax_selected(row, sel):
    """exp(l - max) / sum over the selected logits, in Python floats."""
    m = max(float(row[e]) for e in sel)
    ex = [math.exp(float(row[e]) - m) for e in sel]
    s = sum(ex)
    return [v / s for v in ex]


def test_gate_closed_forms():
    """All-equal logits: the first k experts, each weight 1/k.  Logits
    log(1..8): descending order 7..2 and the renormalised softmax of the
    chosen six."""
    import oracle
    idx, w = oracle.moe_gate(np.zeros((3, 160), np.float32), 3, 160, 6)
    assert (idx == np.arange(6)).all()
    assert np.allclose(w, 1.0 / 6.0, rtol=1e-15, atol=0)
    row = np.log(np.arange(1, 9, dtype=np.float64)).astype(np.float32)
    idx, w = oracle.moe_gate(row[None], 1, 8, 6)
    assert idx[0].tolist() == [7, 6, 5, 4, 3, 2]
    assert np.allclose(w[0], _softmax_selected(row, idx[0]), rtol=1e-14, atol=0)


def test_gate_ties_go_to_the_lower_index():
    import oracle
    row = np.array([[5, 3, 3, 3, 1, 1]], np.float32)
    assert oracle.moe_gate(row, 1, 6, 3)[0][0].tolist() == [0, 1, 2]
    assert oracle.moe_gate(row, 1, 6, 5)[0][0].tolist() == [0, 1, 2, 3, 4]
    assert oracle.moe_gate(np.array([[1, 2, 2]], np.float32), 1, 3, 1)[0][0].tolist() == [1]


def test_gate_matches_stable_sort():
    """Brute force: the chosen experts are a stable descending sort of the
    logits (duplicates included), and the weights the softmax over them."""
    import oracle
    T, E, k = 64, 160, 6
    logits = si.router_logits(T, E, seed=5)
    logits[::3, 10] = logits[::3, 20]          # exact duplicates
    logits[1::4, :8] = logits[1::4, 8:16]
    idx, w = oracle.moe_gate(logits, T, E, k)
    ref = np.argsort(-logits, axis=1, kind="stable")[:, :k]
    assert np.array_equal(idx, ref)
    for t in range(T):
        assert np.allclose(w[t], _softmax_selected(logits[t], idx[t]), rtol=1e-14, atol=0)


def test_gate_large_logits_stay_finite():
    """The max subtraction keeps exp finite for logits near 1000."""
    import oracle
    row = np.array([[1000, 1001, 1002, 990, 1003, 998, 1001, 997]], np.float32)
    idx, w = oracle.moe_gate(row, 1, 8, 4)
    assert idx[0].tolist() == [4, 2, 1, 6]
    assert np.isfinite(w).all()
    assert np.allclose(w[0], _softmax_selected(row[0], idx[0]), rtol=1e-14, atol=0)


# ---------------------------------------------------------------- MoE block

def _block_case(T=3, E=8, H=64, I=32, Is=48, seed=9):
    x = si.activations_bf16(T, H, seed=seed)
    logits = si.router_logits(T, E, seed=seed)
    Wg, Wu, Wd = si.moe_weights(E, H, I, seed=seed)
    Sg, Su, Sd = (a[0] for a in si.moe_weights(1, H, Is, seed=seed + 100))
    return x, logits, Wg, Wu, Wd, Sg, Su, Sd


def test_block_shared_term_is_the_shared_expert():
    """block(with shared) - block(without) = the shared expert alone, run as
    one expert taken by every token with weight 1."""
    import oracle
    T, topk, E, H, I, Is = 3, 6, 8, 64, 32, 48
    x, logits, Wg, Wu, Wd, Sg, Su, Sd = _block_case(T, E, H, I, Is)
    with_s, _, idx, w = oracle.moe_block(x, logits, Wg, Wu, Wd, T, topk, E, H, I, Sg, Su, Sd, Is)
    without, _, idx2, w2 = oracle.moe_block(x, logits, Wg, Wu, Wd, T, topk, E, H, I)
    assert np.array_equal(idx, idx2) and np.array_equal(w, w2)
    shared, _, _ = oracle.moe(x, Sg[None], Su[None], Sd[None], np.zeros((T, 1), np.int32),
                              np.ones((T, 1), np.float32), T, 1, 1, H, Is)
    assert np.allclose(with_s - without, shared, rtol=1e-12, atol=1e-12)


def test_block_identical_experts_collapse():
    """With every routed expert the same matrices, the renormalised weights
    sum to one and the routed sum is that one expert's output."""
    import oracle
    T, topk, E, H, I = 4, 6, 8, 64, 32
    x, logits, Wg, Wu, Wd, *_ = _block_case(T, E, H, I)
    Wg1, Wu1, Wd1 = (np.repeat(a[:1], E, axis=0) for a in (Wg, Wu, Wd))
    out, _, _, w = oracle.moe_block(x, logits, Wg1, Wu1, Wd1, T, topk, E, H, I)
    assert np.allclose(w.sum(axis=1), 1.0, rtol=1e-15, atol=0)
    one, _, _ = oracle.moe(x, Wg[:1], Wu[:1], Wd[:1], np.zeros((T, 1), np.int32),
                           np.ones((T, 1), np.float32), T, 1, 1, H, I)
    assert np.allclose(out, one, rtol=1e-12, atol=1e-12)


def test_block_expert_relabelling():
    """Permuting the experts together with their logit columns changes nothing."""
    import oracle
    T, topk, E, H, I, Is = 3, 6, 8, 64, 32, 48
    x, logits, Wg, Wu, Wd, Sg, Su, Sd = _block_case(T, E, H, I, Is)
    perm = si.rng(9, 77).permutation(E)
    a, _, _, _ = oracle.moe_block(x, logits, Wg, Wu, Wd, T, topk, E, H, I, Sg, Su, Sd, Is)
    b, _, _, _ = oracle.moe_block(x, logits[:, perm], Wg[perm], Wu[perm], Wd[perm], T, topk, E,
                                  H, I, Sg, Su, Sd, Is)
    assert np.allclose(a, b, rtol=1e-12, atol=1e-12)


# ---------------------------------------------------------------- encoder

def test_fp16_encode_matches_numpy(oracle_lib):
    """fp64 -> binary16 nearest-even equals numpy's cast: every fp16 value,
    random fp32 values over the whole range, exact ties, the overflow edge."""
    codes = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    vals = codes.view(np.float16).astype(np.float64)
    for c in range(65536):
        if not math.isnan(vals[c]):
            assert oracle_lib.f64_to_fp16(float(vals[c])) == c, hex(c)
    g = np.random.default_rng(4)
    xs = np.concatenate([
        (g.standard_normal(3000) * np.exp2(g.integers(-30, 17, 3000))).astype(np.float32),
        np.array([65504.0, 65519.99, 65520.0, 1e6, -65520.0, 2.0 ** -25, 2.0 ** -26, 3e-8],
                 np.float32)])
    # ties: the midpoint of two neighbouring fp16 values, both parities
    h = np.array([0x3C00, 0x3C01, 0x0401, 0x0002, 0x7BFE], np.uint16).view(np.float16)
    mids = ((h.astype(np.float64) + np.nextafter(h, np.float16(np.inf)).astype(np.float64)) / 2)
    for x in list(xs.astype(np.float64)) + list(mids):
        with np.errstate(over="ignore"):
            want = int(np.array([x]).astype(np.float16).view(np.uint16)[0])
        assert oracle_lib.f64_to_fp16(float(x)) == want, x


def _codes(B, K, N):
    nb = (N + 31) // 32
    blk = B.reshape(K, nb, 18)
    q = np.empty((K, nb, 32), np.int64)
    q[:, :, 0::2] = blk[:, :, 2:] & 0xF
    q[:, :, 1::2] = blk[:, :, 2:] >> 4
    d = blk[:, :, 0].astype(np.uint16) | (blk[:, :, 1].astype(np.uint16) << 8)
    return q, d


def test_quantize_closed_forms():
    import oracle
    # largest magnitude negative: d = 1/8, codes are the pattern itself
    pat = np.array(list(range(16)) * 2)
    W = ((pat - 8) / 8.0).astype(np.float32)[None]
    q, d = _codes(oracle.quantize(W, 1, 32), 1, 32)
    assert q[0, 0].tolist() == pat.tolist() and d[0, 0] == 0x3000
    # largest magnitude positive: d = -1/8 (negative scale), 1 -> code 0
    W = np.zeros((1, 32), np.float32)
    W[0, :4] = [1.0, 0.5, -0.25, 0.0]
    q, d = _codes(oracle.quantize(W, 1, 32), 1, 32)
    assert d[0, 0] == 0xB000 and q[0, 0, :4].tolist() == [0, 4, 10, 8]
    # all zeros: scale -0, every code 8
    q, d = _codes(oracle.quantize(np.zeros((2, 64), np.float32), 2, 64), 2, 64)
    assert (q == 8).all() and (d == 0x8000).all()
    # a half step rounds up: -0.4375 = -3.5 steps of 1/8 -> code 5
    W = np.zeros((1, 32), np.float32)
    W[0, 0], W[0, 1] = -1.0, -0.4375
    q, _ = _codes(oracle.quantize(W, 1, 32), 1, 32)
    assert q[0, 0, 1] == 5
    # padding columns (>= N) hold code 8
    q, _ = _codes(oracle.quantize(np.ones((1, 40), np.float32), 1, 40), 1, 40)
    assert (q[0, 1, 8:] == 8).all() and (q[0, 1, :8] == 0).all()


def test_quantize_matches_fp32_restatement():
    """The codes equal a numpy fp32 restatement of the same rule (largest
    magnitude first-on-ties, d = m/-8, trunc(w*(1/d) + 8.5) capped at 15)."""
    import oracle
    K, N = 37, 200
    W = (si.rng(8, 1).standard_normal((K, N)) * 0.02).astype(np.float32)
    W[3, 64:96] = 0.0
    W[5, 40], W[5, 41] = 0.05, -0.05             # equal magnitudes: the first wins
    q, d = _codes(oracle.quantize(W, K, N), K, N)
    nb = (N + 31) // 32
    Wp = np.zeros((K, nb * 32), np.float32)
    Wp[:, :N] = W
    Wb = Wp.reshape(K, nb, 32)
    first = np.argmax(np.abs(Wb) == np.abs(Wb).max(axis=2, keepdims=True), axis=2)
    m = np.take_along_axis(Wb, first[..., None], axis=2)[..., 0]
    dd = (m / np.float32(-8.0)).astype(np.float32)
    with np.errstate(divide="ignore"):
        idd = np.where(dd != 0, np.float32(1.0) / dd, np.float32(0.0)).astype(np.float32)
    t = (Wb * idd[..., None]).astype(np.float32)
    t = (t + np.float32(8.5)).astype(np.float32)
    qq = np.minimum(t.astype(np.int64), 15)
    col = np.arange(nb * 32).reshape(nb, 32)
    qq[:, col >= N] = 8
    assert np.array_equal(q, qq)
    assert np.array_equal(d, dd.astype(np.float16).view(np.uint16))


def test_quantize_round_trip_bound():
    """Dequantising the codes gives back each weight within half a step of
    the fp32 scale (a full step where code 16 would be needed and 15 is
    stored) plus 8 times the scale's fp16 rounding."""
    import oracle
    K, N = 64, 320
    W = (si.rng(9, 1).standard_normal((K, N)) * 0.05).astype(np.float32)
    B = oracle.quantize(W, K, N)
    R = oracle.dequant_f32(B, K, N).astype(np.float64)
    nb = N // 32
    Wb = W.astype(np.float64).reshape(K, nb, 32)
    d32 = -np.abs(Wb).max(axis=2) * np.sign(np.take_along_axis(
        Wb, np.abs(Wb).argmax(axis=2)[..., None], axis=2)[..., 0]) / 8.0
    q, dh = _codes(B, K, N)
    d16 = dh.view(np.float16).astype(np.float64)
    steps = Wb / d32[..., None]                 # w in units of the fp32 scale
    half = np.where(steps > 7.5, 1.0, 0.5)      # capped at code 15
    bound = half * np.abs(d32)[..., None] + 8 * np.abs(d32 - d16)[..., None] + 1e-12
    err = np.abs(R.reshape(K, nb, 32) - Wb)
    assert (err <= bound * 1.000001).all()
    assert (steps > 7.5).any()                  # the capped case occurs in the data
