"""GPU routed experts (KTransformers DeepSeek-V2 page, «优化三», «规则二») against
the fp64 oracle, with the oracle's per-element tolerance (the single-matmul
bound 1e-3*sum|a*w| + 1e-6 carried through gate/up, SiLU*up, down and the
weighted sum)."""

import numpy as np
import pytest

import oracle
import seeded_inputs as si
from gpu_util import device, to_dev, torch

import quantized_weight_q4_gb300 as q4

pytestmark = pytest.mark.gpu


def make(T, topk, E, H, I, seed):
    Wg = np.stack([si.q4_weights(H, I, seed, 1000 + e) for e in range(E)])
    Wu = np.stack([si.q4_weights(H, I, seed, 2000 + e) for e in range(E)])
    Wd = np.stack([si.q4_weights(I, H, seed, 3000 + e) for e in range(E)])
    x = si.activations_bf16(T, H, seed)
    idx, w = si.routing(T, E, topk, seed)
    return x, Wg, Wu, Wd, idx, w


def run(x, Wg, Wu, Wd, idx, w, T, topk, E, H, I, dev_weights=None):
    out = torch.empty((T, H), dtype=torch.float32, device=device())
    if dev_weights is None:
        dev_weights = (to_dev(Wg), to_dev(Wu), to_dev(Wd))
    q4.q4_moe_experts_ex(out, to_dev(x), *dev_weights, to_dev(idx), to_dev(w), T, topk, E, H, I)
    torch.cuda.synchronize()
    return out.cpu().numpy().astype(np.float64)


def check(got, ref, tol, what):
    err = np.abs(got - ref)
    bad = ~(err <= tol)
    assert not bad.any(), f"{what}: {bad.sum()} out of tolerance; max excess {np.max(err - tol)}"


@pytest.mark.parametrize("T,topk,E,H,I", [
    (1, 1, 1, 32, 32), (1, 2, 3, 64, 96), (2, 3, 5, 256, 64), (5, 6, 8, 512, 160),
    (3, 2, 16, 300, 100), (9, 4, 7, 1024, 256),
])
def test_moe_small(T, topk, E, H, I):
    x, Wg, Wu, Wd, idx, w = make(T, topk, E, H, I, seed=T + E)
    got = run(x, Wg, Wu, Wd, idx, w, T, topk, E, H, I)
    ref, tol, _ = oracle.moe(x, Wg, Wu, Wd, idx, w, T, topk, E, H, I)
    check(got, ref, tol, f"T={T} topk={topk} E={E} H={H} I={I}")
    assert q4.q4_get_device_status() == q4.Q4_OK


def test_moe_invalid_index_is_skipped_and_flagged():
    T, topk, E, H, I = 3, 3, 6, 256, 96
    x, Wg, Wu, Wd, idx, w = make(T, topk, E, H, I, seed=4)
    idx = idx.copy()
    idx[0, 1] = E
    idx[2, 0] = -3
    got = run(x, Wg, Wu, Wd, idx, w, T, topk, E, H, I)
    ref, tol, _ = oracle.moe(x, Wg, Wu, Wd, idx, w, T, topk, E, H, I)
    check(got, ref, tol, "invalid slots")
    assert q4.q4_get_device_status() == q4.Q4_ERR_DEVICE
    assert q4.q4_last_device_flags() & q4.Q4_DEVERR_INDEX
    assert q4.q4_get_device_status() == q4.Q4_OK   # the word was cleared


def test_moe_all_tokens_one_expert():
    """Every token routes every slot-0 to one expert: the largest token list."""
    T, topk, E, H, I = 12, 2, 4, 512, 128
    x, Wg, Wu, Wd, idx, w = make(T, topk, E, H, I, seed=6)
    idx = idx.copy()
    idx[:, 0] = 2
    idx[:, 1] = np.where(idx[:, 1] == 2, 3, idx[:, 1])
    got = run(x, Wg, Wu, Wd, idx, w, T, topk, E, H, I)
    ref, tol, _ = oracle.moe(x, Wg, Wu, Wd, idx, w, T, topk, E, H, I)
    check(got, ref, tol, "one expert for all")


@pytest.fixture(scope="module")
def deepseek_v2_experts():
    """E = 160 experts, H = 5120, I = 1536 (2.1 GB of Q4_0 weights on the device)."""
    E, H, I = 160, 5120, 1536
    host = si.moe_weights(E, H, I, seed=0)
    dev = tuple(to_dev(a) for a in host)
    return E, H, I, host, dev


@pytest.mark.parametrize("T", [1, 32])
def test_moe_deepseek_v2_shape(T, deepseek_v2_experts):
    """Routed experts at the DeepSeek-V2 shape, top-6 of 160; the oracle checks
    every output of up to 4 sampled tokens (all tokens run on the GPU)."""
    E, H, I, (Wg, Wu, Wd), dev_w = deepseek_v2_experts
    topk = 6
    x = si.activations_bf16(T, H, seed=T)
    idx, w = si.routing(T, E, topk, seed=T)
    got = run(x, Wg, Wu, Wd, idx, w, T, topk, E, H, I, dev_weights=dev_w)
    toks = sorted(set([0, T - 1] + list(si.rng(T, 7).choice(T, size=min(T, 2), replace=False))))
    for t in toks:
        ref, tol, _ = oracle.moe(x[t:t + 1], Wg, Wu, Wd, idx[t:t + 1], w[t:t + 1], 1, topk, E, H, I)
        check(got[t:t + 1], ref, tol, f"T={T} token {t}")
    assert q4.q4_get_device_status() == q4.Q4_OK


def test_moe_after_gemv_shares_library_workspace():
    """A GEMV and the expert path, back to back on the library-owned workspace."""
    from test_gpu_gemv import run as gemv_run
    M, K, N = 2, 300, 520
    A = si.activations_f32(M, K, seed=0)
    B = si.q4_weights(K, N, seed=0)
    gemv_run(A, B, M, N, K)
    T, topk, E, H, I = 2, 3, 5, 256, 64
    x, Wg, Wu, Wd, idx, w = make(T, topk, E, H, I, seed=1)
    for _ in range(2):
        got = run(x, Wg, Wu, Wd, idx, w, T, topk, E, H, I)
        ref, tol, _ = oracle.moe(x, Wg, Wu, Wd, idx, w, T, topk, E, H, I)
        check(got, ref, tol, "after gemv")
        C = gemv_run(A, B, M, N, K)
        C64, S = oracle.matmul(A, B, M, N, K)
        assert np.all(np.abs(C.cpu().numpy() - C64) <= 1e-3 * S + 1e-6)


def test_moe_every_slot_invalid_gives_zeros():
    """No valid routing entry at all: no expert runs, out is exactly zero (the
    oracle's value), and the index error is flagged."""
    T, topk, E, H, I = 2, 3, 4, 256, 64
    x, Wg, Wu, Wd, idx, w = make(T, topk, E, H, I, seed=6)
    idx = np.full_like(idx, -1)
    out = torch.full((T, H), 7.0, dtype=torch.float32, device=device())
    q4.q4_moe_experts_ex(out, to_dev(x), to_dev(Wg), to_dev(Wu), to_dev(Wd), to_dev(idx),
                         to_dev(w), T, topk, E, H, I)
    torch.cuda.synchronize()
    assert not out.any()
    assert q4.q4_get_device_status() == q4.Q4_ERR_DEVICE
    assert q4.q4_last_device_flags() & q4.Q4_DEVERR_INDEX


@pytest.mark.parametrize("T", [1, 5])
def test_moe_captured_on_a_fresh_stream_equals_eager(T):
    """Captured into a CUDA graph on a stream that has seen no eager call, and
    then called eagerly on it: bit-identical outputs, within the oracle's
    tolerance."""
    topk, E, H, I = 3, 6, 512, 96
    x, Wg, Wu, Wd, idx, w = make(T, topk, E, H, I, seed=20 + T)
    d = [to_dev(a) for a in (x, Wg, Wu, Wd, idx, w)]
    ws = torch.zeros(q4.q4_moe_workspace_size(T, topk, E, H, I), dtype=torch.uint8,
                     device=device())
    s = torch.cuda.Stream()
    cap = torch.empty((T, H), dtype=torch.float32, device=device())
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        q4.q4_moe_experts_ex(cap, *d, T, topk, E, H, I, workspace=ws, stream=s)
    g.replay()
    torch.cuda.synchronize()
    eager = torch.empty_like(cap)
    with torch.cuda.stream(s):
        q4.q4_moe_experts_ex(eager, *d, T, topk, E, H, I, workspace=ws, stream=s)
    s.synchronize()
    assert q4.q4_get_device_status() == q4.Q4_OK
    assert torch.equal(cap, eager)
    ref, tol, _ = oracle.moe(x, Wg, Wu, Wd, idx, w, T, topk, E, H, I)
    check(eager.cpu().numpy().astype(np.float64), ref, tol, f"captured and eager T={T}")
