"""The prefill GEMM's shared last round (q4_matmul_bf16_tiles, and
q4_matmul_ex for K >= 1024, with M > 128 and bf16 A; C++ DeepSeek engine
page §5.2, a prompt's tokens as one batched matmul).

The 256 x 256 output tiles that do not fill a whole round over the SMs have
their K steps, taken tile after tile as one range, cut into equal parts over
up to four CTAs per tile.  The part holding a tile's last K step adds the
earlier parts' fp32 partial tiles in K order to its own accumulator and
stores C.  Only the summation order differs from one accumulator per tile, so the
bf16-tile oracle's tolerance (1e-4 * sum|a*bf16(w)| + 1e-6) still holds, and
the bound against the exact product (2^-8 + 1e-4) * S + 1e-6.  The tail runs
when the call has the tail's tickets and partial tiles: the caller's
workspace (q4_matmul_workspace_size bytes, zero before the first call, its
tickets left zero by every call), else, eagerly, the stream's library
scratch; a call captured without a workspace runs every tile whole.
"""

import numpy as np
import pytest

import oracle
import seeded_inputs as si
from gpu_util import device, to_dev, to_host64, torch
from test_gpu_gemm import assert_exact_bound, assert_tile_tol

import quantized_weight_q4_gb300 as q4

pytestmark = pytest.mark.gpu


def sms():
    return torch.cuda.get_device_properties(device()).multi_processor_count


def tail_ctas(M, K, N):
    """CTAs sharing the last round, as the library plans it: the leftover
    tiles' K steps over up to 4 CTAs per tile, at most one CTA per SM and one
    K step per CTA; 0 when a part plus about 6 K steps of partial traffic is
    not shorter than a whole tile."""
    tiles = -(-M // 256) * -(-N // 256)
    ks = -(-K // 64)
    G = sms()
    rem = tiles % G
    if rem == 0:
        return 0
    T = rem * ks
    ctas = min(G, 4 * rem, T)
    return ctas if -(-T // ctas) + 6 <= ks else 0


def run(A, B, M, N, K, workspace=None, stream=None):
    """The tensor-core GEMM itself (q4_matmul_bf16_tiles: any K; q4_matmul_ex
    sends K < 1024 to the exact GEMV)."""
    C = torch.empty((M, N), dtype=torch.float32, device=device())
    q4.q4_matmul_bf16_tiles(C, A, B, M, N, K, workspace=workspace, stream=stream)
    return C


def sampled_rows(M, seed):
    return np.unique(np.concatenate([si.rng(seed, 1).choice(M, 10, replace=False),
                                     [0, min(255, M - 1), M - 1]]))


# (M, K, N): 153 tiles on 152 SMs (one tile left over: four parts of 4 K
# steps), every tile in the tail (16 tiles, M tail rows: four parts of 20
# steps), 80 of 384 tiles left over with an N tail (N = 12280: the last tile
# 248 columns wide) and a short last K step (K = 1000), and 48 tiles (fewer
# than the SMs) with an M tail
SHAPES = [(2304, 1024, 4352), (384, 5120, 2048), (2048, 1000, 12280), (1000, 2048, 3072)]


@pytest.mark.parametrize("M,K,N", SHAPES)
def test_tail_parity(M, K, N):
    assert tail_ctas(M, K, N) > 0
    A = si.activations_bf16(M, K, seed=M + N)
    B = si.q4_weights(K, N, seed=K)
    ws = torch.zeros(q4.q4_matmul_workspace_size(M, N, K), dtype=torch.uint8, device=device())
    C = run(to_dev(A), to_dev(B), M, N, K, workspace=ws)
    torch.cuda.synchronize()
    assert q4.q4_get_device_status() == q4.Q4_OK
    rows = sampled_rows(M, M + N)
    Ch = to_host64(C)[rows]
    Cb, Sb = oracle.matmul_bf16_tiles(A[rows], B, len(rows), N, K)
    assert_tile_tol(Ch, Cb, Sb, f"tail M={M} K={K} N={N}")
    C64, S = oracle.matmul(A[rows], B, len(rows), N, K)
    assert_exact_bound(Ch, C64, S, f"tail M={M} K={K} N={N}")
    # the tickets are zero again for the next call
    assert not ws[:4 * tail_ctas(M, K, N)].any()


def test_tail_repeats_in_graphs_and_without_workspace():
    """Eager calls on one workspace, the same call replayed from a graph, and
    an eager call on the stream's library scratch: bit-identical (the parts
    and their order depend only on the shape and the SM count).  A call
    captured without a workspace runs every tile whole: within the tile
    tolerance."""
    M, K, N = 2304, 1024, 4352
    A = si.activations_bf16(M, K, seed=77)
    B = si.q4_weights(K, N, seed=77)
    dA, dB = to_dev(A), to_dev(B)
    nbytes = q4.q4_matmul_workspace_size(M, N, K)
    assert nbytes >= tail_ctas(M, K, N) * (4 + 128 * 512 * 4)
    ws = torch.zeros(nbytes, dtype=torch.uint8, device=device())
    c1 = run(dA, dB, M, N, K, workspace=ws)
    c2 = run(dA, dB, M, N, K, workspace=ws)
    c3 = run(dA, dB, M, N, K)   # library scratch
    torch.cuda.synchronize()
    assert q4.q4_get_device_status() == q4.Q4_OK
    assert torch.equal(c1, c2) and torch.equal(c1, c3)
    s = torch.cuda.Stream()
    g_ws = torch.empty_like(c1)
    g_whole = torch.empty_like(c1)
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        q4.q4_matmul_bf16_tiles(g_ws, dA, dB, M, N, K, workspace=ws, stream=s)
        q4.q4_matmul_bf16_tiles(g_whole, dA, dB, M, N, K, stream=s)
    for _ in range(3):
        g_ws.fill_(float("nan"))
        g.replay()
        torch.cuda.synchronize()
        assert q4.q4_get_device_status() == q4.Q4_OK
        assert torch.equal(g_ws, c1)
        assert not ws[:4 * tail_ctas(M, K, N)].any()
    rows = sampled_rows(M, 77)
    Cb, Sb = oracle.matmul_bf16_tiles(A[rows], B, len(rows), N, K)
    assert_tile_tol(to_host64(g_whole)[rows], Cb, Sb, "captured without a workspace")
    assert_tile_tol(to_host64(c1)[rows], Cb, Sb, "tail")


def test_tail_one_hot_rows_exact():
    """One nonzero product per sum: the parts' partial tiles are exact (all
    but one part add zeros), so the tail reproduces the bf16 tile rows bit
    for bit."""
    M, K, N = 384, 5120, 2048
    B = si.q4_weights(K, N, seed=35)
    ks = si.rng(35, 2).choice(K, size=M, replace=False)
    A = np.zeros((M, K), np.float32)
    A[np.arange(M), ks] = 1.0
    ws = torch.zeros(q4.q4_matmul_workspace_size(M, N, K), dtype=torch.uint8, device=device())
    C = run(to_dev(si.f32_to_bf16_bits(A)), to_dev(B), M, N, K, workspace=ws)
    torch.cuda.synchronize()
    assert q4.q4_get_device_status() == q4.Q4_OK
    Wb = oracle.dequant_bf16(B, K, N)
    want = (Wb[ks].astype(np.uint32) << 16).view(np.float32)
    assert np.array_equal(C.cpu().numpy(), want)
