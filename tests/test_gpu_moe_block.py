"""GPU router and MoE block against the oracle.

Router: the chosen experts are compared exactly (both sides decide on the
fp32 logits; the softmax is monotonic), the weights within 2e-6 relative
(fp32 exp and division against fp64).  Block: every output element within
the oracle's chain tolerance, which carries the single-matmul tolerance
through gate/up, SiLU, down and the weighted sums, plus 2e-6*|w_k|*|y_k| for
the fp32 router weights.
"""

import numpy as np
import pytest

import oracle
import seeded_inputs as si
from gpu_util import device, to_dev, to_host64, torch

import quantized_weight_q4_gb300 as q4

pytestmark = pytest.mark.gpu


def gate(logits, T, E, topk):
    idx = torch.empty((T, topk), dtype=torch.int32, device=device())
    w = torch.empty((T, topk), dtype=torch.float32, device=device())
    q4.q4_moe_gate(idx, w, to_dev(logits), T, E, topk)
    torch.cuda.synchronize()
    return idx.cpu().numpy(), w.cpu().numpy().astype(np.float64)


def check_gate(logits, T, E, topk, what):
    gi, gw = gate(logits, T, E, topk)
    oi, ow = oracle.moe_gate(logits, T, E, topk)
    assert np.array_equal(gi, oi), what
    assert np.all(np.abs(gw - ow) <= 2e-6 * ow + 1e-7), what


@pytest.mark.parametrize("T,E,topk", [(1, 160, 6), (32, 160, 6), (257, 160, 6), (5, 7, 7),
                                      (9, 1024, 16), (3, 33, 1), (64, 64, 8)])
def test_gate_parity(T, E, topk):
    check_gate(si.router_logits(T, E, seed=T * E + topk), T, E, topk, f"T={T} E={E} k={topk}")


def test_gate_ties_and_large_logits():
    T, E = 16, 160
    logits = si.router_logits(T, E, seed=3)
    logits[::2, 5] = logits[::2, 9]                 # exact duplicates
    logits[1::4, :10] = 0.5
    logits[3] = 0.0                                 # all equal
    logits[5] += 1000.0                             # large logits
    check_gate(logits, T, E, 6, "ties")
    gi, gw = gate(np.zeros((1, E), np.float32), 1, E, 6)
    assert gi[0].tolist() == [0, 1, 2, 3, 4, 5]


def test_gate_shape_errors():
    idx = torch.empty((2, 8), dtype=torch.int32, device=device())
    w = torch.empty((2, 8), dtype=torch.float32, device=device())
    lg = torch.zeros((2, 4096), dtype=torch.float32, device=device())
    for E, k in [(4, 8), (2048, 6), (160, 17)]:
        with pytest.raises(q4.Q4Error) as e:
            q4.q4_moe_gate(idx, w, lg, 2, E, k)
        assert e.value.status == q4.Q4_ERR_SHAPE


def run_block(x, logits, W, S, T, topk, E, H, I, Is, workspace=None):
    out = torch.empty((T, H), dtype=torch.float32, device=device())
    dW = [to_dev(a) for a in W]
    dS = [to_dev(a) for a in S] if Is > 0 else [None, None, None]
    q4.q4_moe_block(out, to_dev(x), to_dev(logits), *dW, T, topk, E, H, I, *dS, Is,
                    workspace=workspace)
    torch.cuda.synchronize()
    assert q4.q4_get_device_status() == q4.Q4_OK
    return to_host64(out)


def check_block(T, topk, E, H, I, Is, seed, x_f32=False):
    x = si.activations_f32(T, H, seed=seed) if x_f32 else si.activations_bf16(T, H, seed=seed)
    logits = si.router_logits(T, E, seed=seed)
    W = si.moe_weights(E, H, I, seed=seed)
    S = tuple(a[0] for a in si.moe_weights(1, H, Is, seed=seed + 100)) if Is > 0 else None
    got = run_block(x, logits, W, S, T, topk, E, H, I, Is)
    kw = dict(Sg=S[0], Su=S[1], Sd=S[2], Is=Is) if Is > 0 else {}
    ref, tol, _, _ = oracle.moe_block(x, logits, *W, T, topk, E, H, I, **kw)
    err = np.abs(got - ref)
    bad = ~(err <= tol)
    assert not bad.any(), (f"{bad.sum()} elements out of tolerance, max err/tol "
                           f"{float(np.max(err / tol)):.3g}")
    return float(np.max(err / tol))


# (4, ..., Is = 512): the shared expert's GEMV shape choice tries cluster
# shapes whose failed queries must leave no CUDA error pending for the
# router's launch
@pytest.mark.parametrize("T,topk,E,H,I,Is", [(3, 6, 8, 256, 64, 128), (5, 2, 4, 512, 96, 0),
                                             (32, 6, 16, 256, 64, 64), (1, 6, 160, 512, 128, 256),
                                             (4, 6, 8, 256, 64, 512)])
def test_block_parity(T, topk, E, H, I, Is):
    check_block(T, topk, E, H, I, Is, seed=T + E)


def test_block_fp32_activations():
    check_block(4, 6, 8, 256, 64, 128, seed=17, x_f32=True)


def test_block_deepseek_v2_one_token():
    """DeepSeek-V2-sized block at T = 1: top-6 of 160 experts, H = 5120,
    I = 1536, shared expert Is = 3072; every output element checked."""
    check_block(1, 6, 160, 5120, 1536, 3072, seed=0)


@pytest.mark.parametrize("T", [1, 4])
def test_block_graph_replay_matches_eager(T):
    """Eager, stream and captured calls agree bit for bit, on both shared-
    expert paths (one routed expert at T = 1, dense GEMVs above)."""
    topk, E, H, I, Is = 6, 16, 512, 128, 256
    x = to_dev(si.activations_bf16(T, H, seed=2))
    logits = to_dev(si.router_logits(T, E, seed=2))
    W = [to_dev(a) for a in si.moe_weights(E, H, I, seed=2)]
    S = [to_dev(a[0]) for a in si.moe_weights(1, H, Is, seed=102)]
    eager = torch.empty((T, H), dtype=torch.float32, device=device())
    q4.q4_moe_block(eager, x, logits, *W, T, topk, E, H, I, *S, Is)
    torch.cuda.synchronize()
    out = torch.zeros_like(eager)
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        q4.q4_moe_block(out, x, logits, *W, T, topk, E, H, I, *S, Is, stream=s)
    s.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        q4.q4_moe_block(out, x, logits, *W, T, topk, E, H, I, *S, Is, stream=s)
    out.zero_()
    g.replay()
    torch.cuda.synchronize()
    assert torch.equal(out, eager)


def test_block_workspace_too_small():
    T, topk, E, H, I, Is = 2, 2, 4, 256, 64, 64
    need = q4.q4_moe_block_workspace_size(T, topk, E, H, I, Is)
    assert need >= q4.q4_moe_workspace_size(T, topk, E, H, I)
    small = torch.zeros(need - 256, dtype=torch.uint8, device=device())
    x = to_dev(si.activations_bf16(T, H, seed=1))
    lg = to_dev(si.router_logits(T, E, seed=1))
    W = [to_dev(a) for a in si.moe_weights(E, H, I, seed=1)]
    S = [to_dev(a[0]) for a in si.moe_weights(1, H, Is, seed=101)]
    out = torch.empty((T, H), dtype=torch.float32, device=device())
    with pytest.raises(q4.Q4Error) as e:
        q4.q4_moe_block(out, x, lg, *W, T, topk, E, H, I, *S, Is, workspace=small)
    assert e.value.status == q4.Q4_ERR_WORKSPACE
