"""GPU tensor-core GEMM (q4_matmul_bf16_tiles: bf16 A, M >= 8, the split-K
small-M form up to 128 rows, the persistent prefill form above) against the
oracle, and q4_matmul_ex's choice between it and the exact GEMV.

The path dequantises every weight to a bf16 tile element, bf16_rn((q-8)*d),
and accumulates bf16 x bf16 products in fp32.  Its own oracle is therefore
A . bf16_rn(W) in fp64 (oracle.matmul_bf16_tiles), and parity is checked
against it element by element within 1e-4 * sum|a*bf16(w)| + 1e-6, ten times
tighter than the matmul tolerance (only the fp32 accumulation differs).

Against the exact product A.W each weight carries up to 2^-8 relative
rounding, so the bound that holds at every K is
|gpu - A.W| <= 2^-8 * S + 1e-4 * S + 1e-6 (S = sum|a*w|); at the prefill
size (K = 5120) the matmul tolerance 1e-3 * S + 1e-6 holds as well, because
the rounding errors have random signs and average out over K terms.
Exact cases: one-hot rows reproduce the bf16 tile values bit for bit; the
bf16 output is the fp32 output rounded to nearest even; results repeat.
"""

import numpy as np
import pytest

import oracle
import seeded_inputs as si
from gpu_util import assert_within_matmul_tol, device, to_dev, to_host64, torch

import quantized_weight_q4_gb300 as q4

pytestmark = pytest.mark.gpu


def run(A, B, M, N, K, c_dtype=torch.float32):
    """The tensor-core GEMM (q4_matmul_bf16_tiles) for bf16 A; q4_matmul_ex
    for fp32 A."""
    C = torch.empty((M, N), dtype=c_dtype, device=device())
    if A.dtype == np.uint16:
        q4.q4_matmul_bf16_tiles(C, to_dev(A), to_dev(B), M, N, K)
    else:
        q4.q4_matmul_ex(C, to_dev(A), to_dev(B), M, N, K)
    torch.cuda.synchronize()
    assert q4.q4_get_device_status() == q4.Q4_OK
    return C


def assert_exact_bound(got, C64, S, what):
    """|gpu - A.W| <= 2^-8 * S + 1e-4 * S + 1e-6: bf16 tile rounding plus fp32
    accumulation.  Returns max |err| / S."""
    err = np.abs(got - C64)
    tol = (2.0 ** -8 + 1e-4) * S + 1e-6
    bad = ~(err <= tol)
    if bad.any():
        i = tuple(np.argwhere(bad)[0])
        raise AssertionError(f"{what}: {bad.sum()} elements beyond the bf16 rounding bound, "
                             f"first {i}: gpu {got[i]!r} oracle {C64[i]!r} tol {tol[i]!r}")
    return float(np.max(err / np.maximum(S, 1e-300)))


def assert_tile_tol(got, Cb, Sb, what):
    err = np.abs(got - Cb)
    tol = 1e-4 * Sb + 1e-6
    bad = ~(err <= tol)
    if bad.any():
        i = tuple(np.argwhere(bad)[0])
        raise AssertionError(f"{what}: {bad.sum()} elements beyond the bf16-tile tolerance, "
                             f"first {i}: gpu {got[i]!r} bf16-tile oracle {Cb[i]!r} tol {tol[i]!r}")


# (M, K, N): single and several tiles in M and N, K tails (K % 64 != 0), an N
# tail inside a tile (N = 250) and M tails.
SHAPES = [
    (65, 64, 256), (128, 520, 256), (256, 64, 512), (300, 520, 1000),
    (513, 1000, 250), (700, 1024, 2048),
]


# The split-K small-M form (8 <= M <= 128): K split over a cluster, partial
# sums combined on chip; K tails, N tails and single-step splits.
SMALL_SHAPES = [
    (8, 64, 256), (8, 5120, 1024), (16, 520, 1000), (33, 1000, 250), (64, 2048, 4096),
    (100, 4096, 512), (128, 320, 2048), (9, 128, 256),
]


@pytest.mark.parametrize("M,K,N", SHAPES + SMALL_SHAPES)
def test_gemm_parity(M, K, N):
    A = si.activations_bf16(M, K, seed=M + K)
    B = si.q4_weights(K, N, seed=N)
    C = to_host64(run(A, B, M, N, K))
    Cb, Sb = oracle.matmul_bf16_tiles(A, B, M, N, K)
    assert_tile_tol(C, Cb, Sb, f"M={M} K={K} N={N}")
    C64, S = oracle.matmul(A, B, M, N, K)
    assert_exact_bound(C, C64, S, f"M={M} K={K} N={N}")


def test_one_hot_rows_give_bf16_tiles():
    """Row i of A = e_{k_i}: C row i is the bf16 tile row k_i exactly (one
    nonzero product per sum), which pins the in-kernel dequantisation, the
    swizzled tile layout and the descriptors."""
    M, K, N = 130, 520, 1000
    B = si.q4_weights(K, N, seed=31)
    ks = si.rng(31, 2).choice(K, size=M, replace=False)
    A = np.zeros((M, K), np.float32)
    A[np.arange(M), ks] = 1.0
    C = run(si.f32_to_bf16_bits(A), B, M, N, K).cpu().numpy()
    Wb = oracle.dequant_bf16(B, K, N)
    want = (Wb[ks].astype(np.uint32) << 16).view(np.float32)
    assert np.array_equal(C, want)


def test_golden_tile_blocks_through_gemm():
    """Hand-rounded bf16 tile values (ties to even) come out of the GEMM."""
    import test_oracle_pins as pins
    recs = pins._golden_bf16_blocks()
    K, N, M = 64, 256, 128
    blocks = [blk for _, blk, _ in recs]
    B = np.frombuffer(b"".join(blocks[(k + b) % len(blocks)] for k in range(K) for b in range(8)),
                      np.uint8).reshape(K, 8 * 18)
    A = np.zeros((M, K), np.float32)
    A[np.arange(M), np.arange(M) % K] = 1.0
    C = run(si.f32_to_bf16_bits(A), B, M, N, K).cpu().numpy()
    for i in range(M):
        k = i % K
        for b in range(8):
            want = np.array(recs[(k + b) % len(recs)][2], np.float32)
            assert np.array_equal(C[i, 32 * b:32 * b + 32], want), (i, b)


@pytest.mark.parametrize("M,K,N", [(300, 520, 1000), (2048, 512, 4096)])
def test_bf16_output_is_rounded_fp32(M, K, N):
    A = si.activations_bf16(M, K, seed=3)
    B = si.q4_weights(K, N, seed=3)
    C32 = run(A, B, M, N, K)
    C16 = run(A, B, M, N, K, c_dtype=torch.bfloat16)
    assert torch.equal(C32.to(torch.bfloat16).view(torch.int16), C16.view(torch.int16))


def test_deterministic_and_padding_free():
    M, K, N = 257, 640, 1000
    A = si.activations_bf16(M, K, seed=5)
    B = si.q4_weights(K, N, seed=5)
    Br = si.randomise_padding(B, K, N, seed=5, stream=99)
    c1 = run(A, B, M, N, K)
    c2 = run(A, B, M, N, K)
    c3 = run(A, Br, M, N, K)
    assert torch.equal(c1, c2)
    assert torch.equal(c1, c3)


def test_zero_weights_and_activations():
    M, K, N = 200, 256, 512
    B = si.q4_weights(K, N, seed=2)
    Z = B.reshape(K, -1, 18).copy()
    Z[:, :, 2:] = 0x88
    A = si.activations_bf16(M, K, seed=2)
    assert not run(A, Z.reshape(K, -1), M, N, K).any()
    assert not run(np.zeros((M, K), np.uint16), B, M, N, K).any()


def test_persistent_tiles_more_than_sms():
    """More output tiles than SMs: CTAs loop over several tiles and reuse the
    accumulators.  Sampled rows, every column."""
    M, K, N = 1024, 192, 256 * 48   # 4 x 48 = 192 tiles
    A = si.activations_bf16(M, K, seed=7)
    B = si.q4_weights(K, N, seed=7)
    C = to_host64(run(A, B, M, N, K))
    rows = np.unique(np.concatenate([si.rng(7, 3).choice(M, 12, replace=False), [0, 255, 256, M - 1]]))
    Cb, Sb = oracle.matmul_bf16_tiles(A[rows], B, len(rows), N, K)
    assert_tile_tol(C[rows], Cb, Sb, "persistent")
    C64, S = oracle.matmul(A[rows], B, len(rows), N, K)
    assert_exact_bound(C[rows], C64, S, "persistent")


def test_prefill_2048x5120x12288():
    """The prefill workload: M = 2048 tokens, K = 5120, N = 12288, bf16 A and
    bf16 output.  16 sampled rows (all 12288 columns) against both oracles;
    the bf16 output equals the fp32 output rounded."""
    M, K, N = 2048, 5120, 12288
    A = si.activations_bf16(M, K, seed=0)
    B = si.q4_weights(K, N, seed=0)
    C32 = run(A, B, M, N, K)
    C16 = run(A, B, M, N, K, c_dtype=torch.bfloat16)
    assert torch.equal(C32.to(torch.bfloat16).view(torch.int16), C16.view(torch.int16))
    C = to_host64(C32)
    rows = np.unique(np.concatenate([si.rng(0, 4).choice(M, 14, replace=False), [0, M - 1]]))
    Cb, Sb = oracle.matmul_bf16_tiles(A[rows], B, len(rows), N, K)
    assert_tile_tol(C[rows], Cb, Sb, "prefill")
    C64, S = oracle.matmul(A[rows], B, len(rows), N, K)
    ratio = assert_within_matmul_tol(C[rows], C64, S, "prefill")
    rel = assert_exact_bound(C[rows], C64, S, "prefill")
    print(f"prefill: max |err|/S = {rel:.3e}, max |err|/(1e-3 S + 1e-6) = {ratio:.3e}")


def test_fp32_activations_above_64_rows_use_gemv():
    """fp32 A with M > 64 keeps the split-K GEMV path (the tensor-core GEMM
    takes bf16 A): still within the exact tolerance."""
    M, K, N = 100, 300, 520
    A = si.activations_f32(M, K, seed=9)
    B = si.q4_weights(K, N, seed=9)
    C = to_host64(run(A, B, M, N, K))
    C64, S = oracle.matmul(A, B, M, N, K)
    assert_within_matmul_tol(C, C64, S, "fp32 A, M = 100")


@pytest.mark.parametrize("M", [8, 16, 32, 64])
def test_small_m_bf16_output_and_determinism(M):
    K, N = 5120, 2048
    A = si.activations_bf16(M, K, seed=40 + M)
    B = si.q4_weights(K, N, seed=40)
    c1 = run(A, B, M, N, K)
    c2 = run(A, B, M, N, K)
    c16 = run(A, B, M, N, K, c_dtype=torch.bfloat16)
    assert torch.equal(c1, c2)
    assert torch.equal(c1.to(torch.bfloat16).view(torch.int16), c16.view(torch.int16))


def test_small_m_one_hot_rows_give_bf16_tiles():
    """The split-K combine adds exact zeros from the other splits: one-hot
    rows still reproduce the bf16 tile values bit for bit."""
    M, K, N = 24, 3000, 1000
    B = si.q4_weights(K, N, seed=41)
    ks = si.rng(41, 2).choice(K, size=M, replace=False)
    A = np.zeros((M, K), np.float32)
    A[np.arange(M), ks] = 1.0
    C = run(si.f32_to_bf16_bits(A), B, M, N, K).cpu().numpy()
    Wb = oracle.dequant_bf16(B, K, N)
    assert np.array_equal(C, (Wb[ks].astype(np.uint32) << 16).view(np.float32))


def _sampled_tile_check(C, A, B, M, N, K, seed, what, nsample=24):
    """24 seeded block columns of C against the bf16-tile oracle."""
    nb = si.nblocks(N)
    cols = np.sort(si.rng(seed, 5).choice(nb, size=min(nsample, nb), replace=False))
    Bs = B.reshape(K, nb, 18)[:, cols].reshape(K, -1)
    Cb, Sb = oracle.matmul_bf16_tiles(A, Bs, M, 32 * len(cols), K)
    got = to_host64(C).reshape(M, nb, 32)[:, cols].reshape(M, -1)
    assert_tile_tol(got, Cb, Sb, what)


@pytest.mark.parametrize("M", [8, 32, 40, 64])
def test_small_m_batched_decode_shape(M):
    """K = 5120, N = 12288 (48 column tiles), bf16 A: up to 40 rows the K
    splits of a tile run as independent CTAs (144 of the 152 SMs in one wave)
    and are added through global memory, at 64 rows over a cluster; sampled
    columns against the bf16-tile oracle, and two runs bit-identical."""
    K, N = 5120, 12288
    A = si.activations_bf16(M, K, seed=50 + M)
    B = si.q4_weights(K, N, seed=50)
    c1 = run(A, B, M, N, K)
    c2 = run(A, B, M, N, K)
    assert torch.equal(c1, c2)
    _sampled_tile_check(c1, A, B, M, N, K, M, f"M={M} 5120x12288")


def test_matmul_ex_short_k_takes_the_exact_gemv():
    """bf16 A, M >= 8, K < 1024: q4_matmul_ex runs the exact-dequant GEMV, so
    the stated tolerance holds with no widening; one-hot rows give the exact
    fp32 weights, not their bf16 roundings."""
    M, K, N = 16, 520, 1000
    A = si.activations_bf16(M, K, seed=71)
    B = si.q4_weights(K, N, seed=71)
    C = torch.empty((M, N), dtype=torch.float32, device=device())
    q4.q4_matmul_ex(C, to_dev(A), to_dev(B), M, N, K)
    torch.cuda.synchronize()
    C64, S = oracle.matmul(A, B, M, N, K)
    assert_within_matmul_tol(to_host64(C), C64, S, "M=16 K=520 bf16 A")
    ks = si.rng(71, 2).choice(K, size=M, replace=False)
    H = np.zeros((M, K), np.float32)
    H[np.arange(M), ks] = 1.0
    q4.q4_matmul_ex(C, to_dev(si.f32_to_bf16_bits(H)), to_dev(B), M, N, K)
    torch.cuda.synchronize()
    assert np.array_equal(C.cpu().numpy(), oracle.dequant_f32(B, K, N)[ks])
    assert q4.q4_get_device_status() == q4.Q4_OK


def test_small_m_eager_capture_grow_replay():
    """Eager M = 8, a graph captured at M = 8, eager M = 40 on the same stream
    (which may replace that stream's library scratch), then replays of the
    graph: the captured call holds no library scratch (it combines its splits
    on chip), so every result matches the bf16-tile oracle and repeats."""
    K, N = 5120, 4096
    s = torch.cuda.Stream()
    ins = {}
    for M in (8, 40):
        A = si.activations_bf16(M, K, seed=80 + M)
        ins[M] = (A, to_dev(A))
    B = si.q4_weights(K, N, seed=80)
    dB = to_dev(B)
    outs = {M: torch.empty((M, N), dtype=torch.float32, device=device()) for M in (8, 40)}
    with torch.cuda.stream(s):
        q4.q4_matmul_ex(outs[8], ins[8][1], dB, 8, N, K, stream=s)
    s.synchronize()
    first = outs[8].clone()
    cap = torch.empty((8, N), dtype=torch.float32, device=device())
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        q4.q4_matmul_ex(cap, ins[8][1], dB, 8, N, K, stream=s)
    with torch.cuda.stream(s):
        q4.q4_matmul_ex(outs[40], ins[40][1], dB, 40, N, K, stream=s)
    s.synchronize()
    for _ in range(3):
        g.replay()
    torch.cuda.synchronize()
    assert q4.q4_get_device_status() == q4.Q4_OK
    for M, got in ((8, first), (8, cap), (40, outs[40])):
        Cb, Sb = oracle.matmul_bf16_tiles(ins[M][0], B, M, N, K)
        assert_tile_tol(to_host64(got), Cb, Sb, f"M={M}")
    with torch.cuda.stream(s):
        q4.q4_matmul_ex(outs[8], ins[8][1], dB, 8, N, K, stream=s)
    s.synchronize()
    assert torch.equal(outs[8], first)


@pytest.mark.parametrize("M", [8, 40])
def test_small_m_caller_workspace_in_a_graph(M):
    """A zeroed caller workspace of q4_matmul_workspace_size bytes carries the
    global split's tickets and partial tiles, eagerly and inside a captured
    graph; replays agree with the eager call and the oracle, and leave the
    tickets at zero."""
    K, N = 5120, 12288
    nbytes = q4.q4_matmul_workspace_size(M, N, K)
    assert nbytes > 0
    ws = torch.zeros(nbytes, dtype=torch.uint8, device=device())
    A = si.activations_bf16(M, K, seed=90 + M)
    B = si.q4_weights(K, N, seed=90)
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
    for _ in range(2):
        g.replay()
    torch.cuda.synchronize()
    assert q4.q4_get_device_status() == q4.Q4_OK
    assert torch.equal(cap, eager)
    tickets = ws[:4 * ((N + 255) // 256)].cpu().numpy()
    assert not tickets.any()
    _sampled_tile_check(eager, A, B, M, N, K, M, f"workspace M={M}")


def test_small_m_capture_on_a_fresh_stream():
    """A call captured into a graph never uses library scratch: it takes the
    cluster form.  Both forms match the
    bf16-tile oracle; eager calls on the same stream afterwards repeat
    exactly, and leave every tile ticket at zero (a third call agrees)."""
    M, K, N = 16, 5120, 4096
    A = si.activations_bf16(M, K, seed=61)
    B = si.q4_weights(K, N, seed=61)
    dA, dB = to_dev(A), to_dev(B)
    s = torch.cuda.Stream()
    out = torch.empty((M, N), dtype=torch.float32, device=device())
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        q4.q4_matmul_ex(out, dA, dB, M, N, K, stream=s)
    g.replay()
    torch.cuda.synchronize()
    assert q4.q4_get_device_status() == q4.Q4_OK
    Cb, Sb = oracle.matmul_bf16_tiles(A, B, M, N, K)
    assert_tile_tol(to_host64(out), Cb, Sb, "captured (cluster form)")
    eager = []
    for _ in range(3):
        c = torch.empty((M, N), dtype=torch.float32, device=device())
        with torch.cuda.stream(s):
            q4.q4_matmul_ex(c, dA, dB, M, N, K, stream=s)
        s.synchronize()
        eager.append(c)
    assert q4.q4_get_device_status() == q4.Q4_OK
    assert torch.equal(eager[0], eager[1]) and torch.equal(eager[1], eager[2])
    assert_tile_tol(to_host64(eager[0]), Cb, Sb, "eager (global split)")


# Prefill with more 256 x 256 tiles than SMs and an uneven last round (2048 x
# 5888 = 8 x 23 = 184 tiles; K = 520: nine K steps, the last one short): CTAs
# take several tiles, and each tile's epilogue stages C in shared memory that
# the next tile's B stages reuse (the TMA-store epilogue).
def test_prefill_several_tiles_per_cta():
    M, K, N = 2048, 520, 5888
    A = si.activations_bf16(M, K, seed=21)
    B = si.q4_weights(K, N, seed=21)
    C = run(A, B, M, N, K)
    C2 = run(A, B, M, N, K)
    assert torch.equal(C, C2)
    Ch = to_host64(C)
    rows = np.unique(np.concatenate([si.rng(21, 1).choice(M, 10, replace=False),
                                     [0, 255, 256, 1023, 1024, M - 1]]))
    Cb, Sb = oracle.matmul_bf16_tiles(A[rows], B, len(rows), N, K)
    assert_tile_tol(Ch[rows], Cb, Sb, "several tiles per CTA")
    C64, S = oracle.matmul(A[rows], B, len(rows), N, K)
    assert_exact_bound(Ch[rows], C64, S, "several tiles per CTA")
    C16 = run(A, B, M, N, K, c_dtype=torch.bfloat16)
    assert torch.equal(C.to(torch.bfloat16).view(torch.int16), C16.view(torch.int16))
