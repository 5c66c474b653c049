"""Routed experts of several tokens in one persistent launch (KTransformers
DeepSeek-V2 page, «优化三»: the chosen experts' gate and up, SiLU(g) * u,
down, and the weighted sum of the slots, as small GEMVs).

From 4 tokens up, q4_moe_experts_ex runs the decode-sequence kernel on two
segmented ops: gate and up of every slot s = t * topk + k (expert
topk_idx[s], input x[t]), whose last K slice of each column tile forms
h = SiLU(g) * u there, then down of every slot (input h[s]), each slot
waiting only for its own h; the slot combine follows.  The launch takes its
counters from the workspace's first 64 KB and leaves them zero, so that the
next call (eager or replayed) starts from zero.

Stage by stage, through q4_moe_experts_trace, against fp64 recomputations on
the GPU's own inputs to each stage (g, u and y at 1e-3 * S + 1e-6; h within
the fp32 rounding of SiLU and the product; the slot sum within topk fused
multiply-adds), and the output against the oracle's chain tolerance.
"""

import numpy as np
import pytest

import oracle
import seeded_inputs as si
from gpu_util import device, to_dev, torch
from test_gpu_moe_stages import check_chain, check_stages, make, trace

import quantized_weight_q4_gb300 as q4

pytestmark = pytest.mark.gpu

HEADER = 64 * 1024


# (T, topk, E, H, I): gate/up over one K slice of 1280 rows,
# the column tail inside a slot (I = 768: 1.5 tiles), down over one K slice of
# 768 rows, the output tail (H = 1280: 2.5 tiles), slots sharing experts (E
# small), more slots than experts, topk = 1, I > 4096 (down in two K
# slices, added through partial rows and tickets), the DeepSeek-V2 experts at
# the fewest tokens that take this form (two K slices of 2560 rows), and
# H = 4328 (gate/up in K slices of 2176 and 2152 rows, the last stage 40 rows;
# down's last output tile 232 columns) with I = 256 (one half-width tile)
SHAPES = [(8, 3, 5, 1280, 768), (9, 6, 8, 2048, 512), (16, 1, 3, 512, 256),
          (24, 6, 40, 1024, 1536), (8, 8, 12, 768, 2304), (8, 2, 3, 512, 4608),
          (4, 6, 160, 5120, 1536), (5, 2, 7, 4328, 256)]


@pytest.mark.parametrize("T,topk,E,H,I", SHAPES)
def test_seq_moe_stages(T, topk, E, H, I):
    x, Wg, Wu, Wd, idx, w = make(T, topk, E, H, I, seed=T + 7 * E)
    dW = tuple(to_dev(a) for a in (Wg, Wu, Wd))
    res = trace(x, dW, idx, w, T, topk, E, H, I)
    toks = sorted(set([0, T - 1, T // 2]))
    check_stages(x, Wg, Wu, Wd, idx, w, T, topk, E, H, I, res, toks)
    check_chain(x, Wg, Wu, Wd, idx, w, T, topk, E, H, I, res[0], toks)


def run(out, d, T, topk, E, H, I, ws, stream=None):
    q4.q4_moe_experts_ex(out, *d, T, topk, E, H, I, workspace=ws, stream=stream)


def test_seq_moe_repeated_and_captured_calls_leave_counters_zero():
    """Eager calls, then a graph of two calls replayed three times, on one
    workspace: every result bit-identical, the header zero after each."""
    T, topk, E, H, I = 12, 6, 10, 2048, 768
    x, Wg, Wu, Wd, idx, w = make(T, topk, E, H, I, seed=5)
    d = [to_dev(a) for a in (x, Wg, Wu, Wd, idx, w)]
    ws = torch.zeros(q4.q4_moe_workspace_size(T, topk, E, H, I), dtype=torch.uint8,
                     device=device())
    outs = [torch.full((T, H), float("nan"), dtype=torch.float32, device=device())
            for _ in range(3)]
    for o in outs:
        run(o, d, T, topk, E, H, I, ws)
    torch.cuda.synchronize()
    assert q4.q4_get_device_status() == q4.Q4_OK
    assert not ws[:HEADER].any()
    for o in outs[1:]:
        assert torch.equal(o, outs[0])
    s = torch.cuda.Stream()
    a = torch.empty_like(outs[0])
    b = torch.empty_like(outs[0])
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        run(a, d, T, topk, E, H, I, ws, stream=s)
        run(b, d, T, topk, E, H, I, ws, stream=s)
    for _ in range(3):
        a.fill_(float("nan"))
        b.fill_(float("nan"))
        g.replay()
        torch.cuda.synchronize()
        assert q4.q4_get_device_status() == q4.Q4_OK
        assert torch.equal(a, outs[0]) and torch.equal(b, outs[0])
        assert not ws[:HEADER].any()
    want, tol, _ = oracle.moe(x, Wg, Wu, Wd, idx, w, T, topk, E, H, I)
    assert np.all(np.abs(outs[0].cpu().numpy().astype(np.float64) - want) <= tol)


def test_seq_moe_trace_matches_experts_ex():
    T, topk, E, H, I = 10, 6, 9, 1280, 768
    x, Wg, Wu, Wd, idx, w = make(T, topk, E, H, I, seed=8)
    dW = tuple(to_dev(a) for a in (Wg, Wu, Wd))
    out = trace(x, dW, idx, w, T, topk, E, H, I)[0]
    ref = torch.empty((T, H), dtype=torch.float32, device=device())
    q4.q4_moe_experts_ex(ref, to_dev(x), *dW, to_dev(idx), to_dev(w), T, topk, E, H, I)
    torch.cuda.synchronize()
    assert q4.q4_get_device_status() == q4.Q4_OK
    assert np.array_equal(out, ref.cpu().numpy())


def test_seq_moe_invalid_slots_skipped_and_flagged():
    """Slots whose index lies outside [0, E) read no weights, add nothing and
    leave their trace rows unwritten; the call records Q4_DEVERR_INDEX and
    leaves the counters zero."""
    T, topk, E, H, I = 8, 5, 7, 1280, 512
    x, Wg, Wu, Wd, idx, w = make(T, topk, E, H, I, seed=9)
    idx = idx.copy()
    idx[0, 1] = E
    idx[3, 3] = -1
    dW = tuple(to_dev(a) for a in (Wg, Wu, Wd))
    f = lambda *s: torch.full(s, float("nan"), dtype=torch.float32, device=device())
    out, g, u, h, y = f(T, H), f(T * topk, I), f(T * topk, I), f(T * topk, I), f(T * topk, H)
    ws = torch.zeros(q4.q4_moe_workspace_size(T, topk, E, H, I), dtype=torch.uint8,
                     device=device())
    q4.q4_moe_experts_trace(out, to_dev(x), *dW, to_dev(idx), to_dev(w), T, topk, E, H, I,
                            ws, g, u, h, y)
    torch.cuda.synchronize()
    assert q4.q4_get_device_status() == q4.Q4_ERR_DEVICE
    assert q4.q4_last_device_flags() & q4.Q4_DEVERR_INDEX
    assert not ws[:HEADER].any()
    bad = [0 * topk + 1, 3 * topk + 3]
    for a in (g, u, h, y):
        rows = torch.isnan(a).all(dim=1).cpu().numpy()
        assert list(np.nonzero(rows)[0]) == bad
    # token 0 through the oracle with its valid slots
    keep = [k for k in range(topk) if k != 1]
    want, tol, _ = oracle.moe(x[:1], Wg, Wu, Wd, idx[:1, keep].copy(), w[:1, keep].copy(), 1,
                              len(keep), E, H, I)
    assert np.all(np.abs(out[:1].cpu().numpy().astype(np.float64) - want) <= tol)


def test_seq_moe_every_slot_invalid_gives_zeros():
    T, topk, E, H, I = 8, 3, 4, 512, 256
    x, Wg, Wu, Wd, idx, w = make(T, topk, E, H, I, seed=10)
    idx = np.full_like(idx, E + 3)
    out = torch.full((T, H), float("nan"), dtype=torch.float32, device=device())
    ws = torch.zeros(q4.q4_moe_workspace_size(T, topk, E, H, I), dtype=torch.uint8,
                     device=device())
    q4.q4_moe_experts_ex(out, to_dev(x), to_dev(Wg), to_dev(Wu), to_dev(Wd), to_dev(idx),
                         to_dev(w), T, topk, E, H, I, workspace=ws)
    torch.cuda.synchronize()
    assert q4.q4_get_device_status() == q4.Q4_ERR_DEVICE
    assert not out.any()
    assert not ws[:HEADER].any()


def test_seq_moe_fp32_activations():
    T, topk, E, H, I = 8, 4, 6, 1024, 512
    Wg, Wu, Wd = si.moe_weights(E, H, I, seed=12)
    x = si.activations_f32(T, H, 12)
    idx, w = si.routing(T, E, topk, 12)
    out = torch.empty((T, H), dtype=torch.float32, device=device())
    q4.q4_moe_experts_ex(out, to_dev(x), to_dev(Wg), to_dev(Wu), to_dev(Wd), to_dev(idx),
                         to_dev(w), T, topk, E, H, I)
    torch.cuda.synchronize()
    assert q4.q4_get_device_status() == q4.Q4_OK
    want, tol, _ = oracle.moe(x, Wg, Wu, Wd, idx, w, T, topk, E, H, I)
    assert np.all(np.abs(out.cpu().numpy().astype(np.float64) - want) <= tol)


def test_seq_moe_small_workspace_takes_three_launches():
    """A workspace smaller than q4_moe_workspace_size but large enough for the
    three-launch form (as the 8 MiB of q4_moe_experts_noalloc at 32 tokens)
    runs that form: within the chain tolerance of the oracle."""
    T, topk, E, H, I = 32, 6, 12, 512, 256
    x, Wg, Wu, Wd, idx, w = make(T, topk, E, H, I, seed=14)
    nb = q4.q4_moe_workspace_size(T, topk, E, H, I)
    small = HEADER + T * topk * (H + I) * 4 + 4096
    assert small < nb
    ws = torch.zeros(small, dtype=torch.uint8, device=device())
    out = torch.empty((T, H), dtype=torch.float32, device=device())
    q4.q4_moe_experts_ex(out, to_dev(x), to_dev(Wg), to_dev(Wu), to_dev(Wd), to_dev(idx),
                         to_dev(w), T, topk, E, H, I, workspace=ws)
    torch.cuda.synchronize()
    assert q4.q4_get_device_status() == q4.Q4_OK
    want, tol, _ = oracle.moe(x, Wg, Wu, Wd, idx, w, T, topk, E, H, I)
    assert np.all(np.abs(out.cpu().numpy().astype(np.float64) - want) <= tol)


def test_seq_moe_block_eight_tokens():
    """The MoE block at T = 8: the dense shared expert, then the routed
    experts on the persistent form with the shared rows as the combine's
    addend."""
    T, topk, E, H, I, Is = 8, 6, 12, 1024, 256, 512
    Wg, Wu, Wd = si.moe_weights(E, H, I, seed=13)
    Sg, Su, Sd = (a[0] for a in si.moe_weights(1, H, Is, seed=113))
    x = si.activations_bf16(T, H, seed=13)
    logits = si.router_logits(T, E, seed=13)
    out = torch.empty((T, H), dtype=torch.float32, device=device())
    ws = torch.zeros(q4.q4_moe_block_workspace_size(T, topk, E, H, I, Is), dtype=torch.uint8,
                     device=device())
    q4.q4_moe_block(out, to_dev(x), to_dev(logits), to_dev(Wg), to_dev(Wu), to_dev(Wd), T, topk,
                    E, H, I, to_dev(Sg), to_dev(Su), to_dev(Sd), Is, workspace=ws)
    torch.cuda.synchronize()
    assert q4.q4_get_device_status() == q4.Q4_OK
    assert not ws[:HEADER].any()
    want, tol = oracle.moe_block(x, logits, Wg, Wu, Wd, T, topk, E, H, I, Sg, Su, Sd, Is)[:2]
    assert np.all(np.abs(out.cpu().numpy().astype(np.float64) - want) <= tol)
