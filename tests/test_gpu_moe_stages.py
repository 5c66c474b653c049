"""Routed experts checked stage by stage (KTransformers DeepSeek-V2 page,
«优化三»: gate and up, SiLU(g) * u, down, the weighted sum of the slots;
C++ DeepSeek engine page §8.2: fixed inputs, every stage compared).

q4_moe_experts_trace runs the same kernels as q4_moe_experts_ex and also
returns g, u, h and y.  Each stage is compared with an fp64 recomputation
on the GPU's own input to that stage, so a wrong stage cannot hide behind
the rest of the chain:

  g, u   against oracle.matmul(x_t, W_gate[e]) and (x_t, W_up[e]) at the
         stated single-matmul tolerance 1e-3 * S + 1e-6;
  h      against SiLU(g) * u evaluated in fp64 from the GPU's g and u, within
         the rounding of fp32 exp, division and product, (8 + 2|g|) * 2^-24;
  y      against oracle.matmul(h_gpu, W_down[e]) at 1e-3 * S + 1e-6;
  out    against sum_k w_k * y_k in fp64 from the GPU's y, within the
         rounding of topk fused multiply-adds;

and the output as a whole against the oracle's chain with its per-element
tolerance (the fp32 rounding bound carried through the chain).
"""

import numpy as np
import pytest

import oracle
import seeded_inputs as si
from gpu_util import assert_within_matmul_tol, device, to_dev, torch

import quantized_weight_q4_gb300 as q4

pytestmark = pytest.mark.gpu

U = 2.0 ** -24


def trace(x, dW, idx, w, T, topk, E, H, I):
    f = lambda *s: torch.full(s, float("nan"), dtype=torch.float32, device=device())
    out, g, u, h, y = f(T, H), f(T * topk, I), f(T * topk, I), f(T * topk, I), f(T * topk, H)
    ws = torch.zeros(q4.q4_moe_workspace_size(T, topk, E, H, I), dtype=torch.uint8,
                     device=device())
    q4.q4_moe_experts_trace(out, to_dev(x), *dW, to_dev(idx), to_dev(w), T, topk, E, H, I,
                            ws, g, u, h, y)
    torch.cuda.synchronize()
    assert q4.q4_get_device_status() == q4.Q4_OK
    return [a.cpu().numpy() for a in (out, g, u, h, y)]


def check_stages(x, Wg, Wu, Wd, idx, w, T, topk, E, H, I, res, tokens):
    out, g, u, h, y = res
    silu = np.vectorize(oracle.silu)
    for t in tokens:
        xt = x[t:t + 1]
        for k in range(topk):
            s, e = t * topk + k, int(idx[t, k])
            what = f"token {t} slot {k} expert {e}"
            g64, Sg = oracle.matmul(xt, Wg[e], 1, I, H)
            u64, Su = oracle.matmul(xt, Wu[e], 1, I, H)
            assert_within_matmul_tol(g[s:s + 1].astype(np.float64), g64, Sg, "g " + what)
            assert_within_matmul_tol(u[s:s + 1].astype(np.float64), u64, Su, "u " + what)
            gg, uu = g[s].astype(np.float64), u[s].astype(np.float64)
            hh = silu(gg) * uu
            err = np.abs(h[s].astype(np.float64) - hh)
            assert (err <= (8.0 + 2.0 * np.abs(gg)) * U * np.abs(hh) + 1e-30).all(), "h " + what
            y64, Sy = oracle.matmul(h[s:s + 1], Wd[e], 1, H, I)
            assert_within_matmul_tol(y[s:s + 1].astype(np.float64), y64, Sy, "y " + what)
        yw = w[t].astype(np.float64)[:, None] * y[t * topk:(t + 1) * topk].astype(np.float64)
        err = np.abs(out[t].astype(np.float64) - yw.sum(axis=0))
        assert (err <= 2 * topk * U * np.abs(yw).sum(axis=0) + 1e-30).all(), f"combine token {t}"


def check_chain(x, Wg, Wu, Wd, idx, w, T, topk, E, H, I, out, tokens):
    for t in tokens:
        ref, tol, _ = oracle.moe(x[t:t + 1], Wg, Wu, Wd, idx[t:t + 1], w[t:t + 1], 1, topk, E,
                                 H, I)
        err = np.abs(out[t:t + 1].astype(np.float64) - ref)
        bad = ~(err <= tol)
        assert not bad.any(), f"token {t}: {bad.sum()} outputs beyond the chain tolerance"


def make(T, topk, E, H, I, seed):
    Wg, Wu, Wd = si.moe_weights(E, H, I, seed=seed)
    x = si.activations_bf16(T, H, seed)
    idx, w = si.routing(T, E, topk, seed)
    return x, Wg, Wu, Wd, idx, w


@pytest.mark.parametrize("T,topk,E,H,I", [
    (1, 1, 1, 32, 32), (2, 3, 5, 256, 64), (5, 6, 8, 512, 160), (3, 2, 16, 300, 100),
    (9, 4, 7, 1024, 256), (12, 6, 20, 2048, 512),
])
def test_stages_small(T, topk, E, H, I):
    x, Wg, Wu, Wd, idx, w = make(T, topk, E, H, I, seed=T + 11 * E)
    dW = tuple(to_dev(a) for a in (Wg, Wu, Wd))
    res = trace(x, dW, idx, w, T, topk, E, H, I)
    check_stages(x, Wg, Wu, Wd, idx, w, T, topk, E, H, I, res, range(T))
    check_chain(x, Wg, Wu, Wd, idx, w, T, topk, E, H, I, res[0], range(T))


def test_trace_matches_experts_ex():
    """The traced call is the same computation: its output is bit-identical
    to q4_moe_experts_ex's."""
    T, topk, E, H, I = 4, 3, 6, 512, 96
    x, Wg, Wu, Wd, idx, w = make(T, topk, E, H, I, seed=3)
    dW = tuple(to_dev(a) for a in (Wg, Wu, Wd))
    out = trace(x, dW, idx, w, T, topk, E, H, I)[0]
    ref = torch.empty((T, H), dtype=torch.float32, device=device())
    q4.q4_moe_experts_ex(ref, to_dev(x), *dW, to_dev(idx), to_dev(w), T, topk, E, H, I)
    torch.cuda.synchronize()
    assert np.array_equal(out, ref.cpu().numpy())


@pytest.fixture(scope="module")
def deepseek_v2():
    """E = 160 experts, H = 5120, I = 1536 (2.1 GB of Q4_0 weights)."""
    E, H, I = 160, 5120, 1536
    host = si.moe_weights(E, H, I, seed=0)
    return E, H, I, host, tuple(to_dev(a) for a in host)


@pytest.mark.parametrize("T", [1, 32])
def test_stages_deepseek_v2(T, deepseek_v2):
    """Top-6 of 160 at H = 5120, I = 1536: every stage of three sampled tokens
    (all of them at T = 1), and their outputs against the chain tolerance."""
    E, H, I, (Wg, Wu, Wd), dW = deepseek_v2
    topk = 6
    x = si.activations_bf16(T, H, seed=T)
    idx, w = si.routing(T, E, topk, seed=T)
    res = trace(x, dW, idx, w, T, topk, E, H, I)
    toks = sorted(set([0, T - 1, int(si.rng(T, 9).integers(0, T))]))
    check_stages(x, Wg, Wu, Wd, idx, w, T, topk, E, H, I, res, toks)
    check_chain(x, Wg, Wu, Wd, idx, w, T, topk, E, H, I, res[0], toks)
