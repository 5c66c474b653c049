"""Pins of the routed-expert chain tolerance (oracle.moe's tol) at the
DeepSeek-V2 shape of the KTransformers page («优化三»: 160 routed experts,
6 active per token; H = 5120, I = 1536).

The tolerance must admit a correct fp32 evaluation of the chain and reject
plausible mistakes: an all-zero output, a dropped slot, a wrong expert, two
slots' experts exchanged.  Only the experts a token uses are generated (with
the streams they have in the full 160-expert stack), so these run on the CPU.
"""

import numpy as np
import pytest

import oracle
import seeded_inputs as si

E, H, I, TOPK = 160, 5120, 1536, 6


def token_problem(T, t, extra=()):
    """Token t of the seeded T-token routing, with its experts (plus `extra`)
    as a compact stack and the routing relabelled to it."""
    x = si.activations_bf16(T, H, seed=T)[t:t + 1]
    idx, w = si.routing(T, E, TOPK, seed=T)
    idx, w = idx[t:t + 1], w[t:t + 1]
    chosen = sorted(set(idx.reshape(-1).tolist()) | set(extra))
    pos = {e: i for i, e in enumerate(chosen)}
    Wg = np.stack([si.q4_weights(H, I, 0, 1000 + e) for e in chosen])
    Wu = np.stack([si.q4_weights(H, I, 0, 2000 + e) for e in chosen])
    Wd = np.stack([si.q4_weights(I, H, 0, 3000 + e) for e in chosen])
    li = np.vectorize(pos.get)(idx).astype(np.int32)
    return x, Wg, Wu, Wd, li, w, pos


def bf16_to_f32(x):
    return (x.astype(np.uint32) << 16).view(np.float32)


def fp32_chain(x, Wg, Wu, Wd, idx, w):
    """The chain evaluated in fp32 with numpy's matmul (blocked fp32 sums) on
    the exact dequantised weights."""
    x32 = bf16_to_f32(x)
    out = np.zeros((1, H), np.float32)
    for k in range(TOPK):
        e = idx[0, k]
        g = x32 @ oracle.dequant_f32(Wg[e], H, I)
        u = x32 @ oracle.dequant_f32(Wu[e], H, I)
        h = (g / (np.float32(1.0) + np.exp(-g)) * u).astype(np.float32)
        y = h @ oracle.dequant_f32(Wd[e], I, H)
        out = out + w[0, k] * y
    return out.astype(np.float64)


def beyond(got, ref, tol):
    return float(np.mean(np.abs(got - ref) > tol))


@pytest.mark.parametrize("T,t", [(1, 0), (32, 0), (32, 17)])
def test_chain_tolerance_at_deepseek_v2_shape(T, t):
    x, Wg, Wu, Wd, idx, w, pos = token_problem(T, t, extra=(159, 158))
    n = len(pos)
    out, tol, _ = oracle.moe(x, Wg, Wu, Wd, idx, w, 1, TOPK, n, H, I)
    # not vacuous: the tolerance is a fraction of the output it bounds
    assert np.median(tol / np.abs(out)) < 0.5
    # a correct fp32 evaluation stays far inside it
    assert beyond(fp32_chain(x, Wg, Wu, Wd, idx, w), out, tol) == 0.0
    # an all-zero output fails on most elements
    assert beyond(np.zeros_like(out), out, tol) > 0.5
    # dropping any one slot fails
    for k in range(TOPK):
        w2 = w.copy()
        w2[0, k] = 0.0
        o2, _, _ = oracle.moe(x, Wg, Wu, Wd, idx, w2, 1, TOPK, n, H, I)
        assert beyond(o2, out, tol) > 0.2, f"slot {k} dropped"
    # a wrong expert in the first and in the last slot fails
    spare = pos[159] if pos[159] not in idx[0] else pos[158]
    for k in (0, TOPK - 1):
        i2 = idx.copy()
        i2[0, k] = spare
        o3, _, _ = oracle.moe(x, Wg, Wu, Wd, i2, w, 1, TOPK, n, H, I)
        assert beyond(o3, out, tol) > 0.5, f"wrong expert in slot {k}"
    # the experts of two slots exchanged (weights kept) fails
    i4 = idx.copy()
    i4[0, 0], i4[0, TOPK - 1] = idx[0, TOPK - 1], idx[0, 0]
    o4, _, _ = oracle.moe(x, Wg, Wu, Wd, i4, w, 1, TOPK, n, H, I)
    assert beyond(o4, out, tol) > 0.2


def test_chain_tolerance_grows_with_the_weights():
    """Scaling every routing weight by 2 scales the output by 2 and the
    tolerance by 2, up to its absolute 1e-6 term."""
    x, Wg, Wu, Wd, idx, w, pos = token_problem(1, 0)
    n = len(pos)
    out, tol, _ = oracle.moe(x, Wg, Wu, Wd, idx, w, 1, TOPK, n, H, I)
    out2, tol2, _ = oracle.moe(x, Wg, Wu, Wd, idx, (2 * w).astype(np.float32), 1, TOPK, n, H, I)
    assert np.allclose(out2, 2 * out, rtol=1e-12, atol=0)
    assert np.allclose(tol2 - 1e-6, 2 * (tol - 1e-6), rtol=1e-9, atol=0)
