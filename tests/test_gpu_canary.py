"""Bounds of every output write, checked with canary bytes.

Each output buffer sits inside a larger allocation whose bytes before and
after it, and the output itself, start as a sentinel pattern (a NaN payload
no kernel produces).  After the call no byte outside the output may have
changed, and every element inside it must have been written.  The cases
cover the tails of each kernel form: N not a multiple of 32 or of the column
tile, M not a multiple of the rows per pass or per MMA tile, K not a multiple
of the stage, for the split-K GEMV, the tensor-core GEMM (both small-M forms
and the prefill form, its shared last round included), bf16 and fp32
outputs, and the routed experts' out in both forms.
(The compute sanitizer is closed on this machine; this is its stand-in for
out-of-bounds stores.)
"""

import numpy as np
import pytest

import seeded_inputs as si
from gpu_util import device, to_dev, torch

import quantized_weight_q4_gb300 as q4

pytestmark = pytest.mark.gpu

PAD = 4096          # guard bytes on each side
SENT32 = 0x7FA5A5A5  # fp32 NaN with a payload the kernels never write
SENT16 = 0x7FA5      # bf16 NaN, likewise


def guarded(n, dtype):
    """(whole buffer, view of n elements at a 256-byte aligned offset PAD in)."""
    es = 4 if dtype == torch.float32 else 2
    total = n * es + 2 * PAD
    raw = torch.empty(total, dtype=torch.uint8, device=device())
    if es == 4:
        raw.view(torch.int32).fill_(SENT32)
    else:
        raw.view(torch.int16).fill_(SENT16 - 65536 if SENT16 > 32767 else SENT16)
    view = raw[PAD:PAD + n * es].view(dtype)
    return raw, view


def check_guard(raw, n, dtype, what):
    es = 4 if dtype == torch.float32 else 2
    b = raw.cpu().numpy()
    pat = np.full(PAD // es, SENT32 if es == 4 else SENT16,
                  dtype=np.uint32 if es == 4 else np.uint16).view(np.uint8)
    assert np.array_equal(b[:PAD], pat), f"{what}: bytes before the output changed"
    assert np.array_equal(b[PAD + n * es:], pat), f"{what}: bytes after the output changed"
    inner = b[PAD:PAD + n * es].view(np.uint32 if es == 4 else np.uint16)
    left = int(np.sum(inner == (SENT32 if es == 4 else SENT16)))
    assert left == 0, f"{what}: {left} output elements never written"


# (M, K, N, a_dtype, c_dtype, entry): GEMV tails, tensor-core small-M (global
# form up to 40 rows, cluster form above), prefill with M and N tails (its
# TMA-store epilogue: boxes of 32 rows clipped at M and N)
CASES = [
    (1, 300, 250, "f32", "f32", "ex"), (3, 517, 1000, "f32", "f32", "ex"),
    (5, 64, 33, "bf16", "bf16", "ex"), (7, 2049, 4000, "bf16", "f32", "ex"),
    (64, 200, 520, "f32", "bf16", "ex"), (2, 16384, 2048, "f32", "f32", "ex"),
    (9, 1024, 250, "bf16", "f32", "tiles"), (33, 5120, 1000, "bf16", "bf16", "tiles"),
    (40, 2048, 4096, "bf16", "f32", "tiles"), (100, 1000, 250, "bf16", "f32", "tiles"),
    (129, 520, 1000, "bf16", "bf16", "tiles"), (300, 2048, 2040, "bf16", "f32", "tiles"),
    (333, 640, 1000, "bf16", "bf16", "ex"),
]


@pytest.mark.parametrize("M,K,N,adt,cdt,entry", CASES)
def test_matmul_writes_exactly_its_output(M, K, N, adt, cdt, entry):
    A = si.activations_bf16(M, K, seed=M) if adt == "bf16" else si.activations_f32(M, K, seed=M)
    B = si.q4_weights(K, N, seed=K)
    ct = torch.float32 if cdt == "f32" else torch.bfloat16
    raw, C = guarded(M * N, ct)
    C = C.view(M, N)
    fn = q4.q4_matmul_ex if entry == "ex" else q4.q4_matmul_bf16_tiles
    fn(C, to_dev(A), to_dev(B), M, N, K)
    torch.cuda.synchronize()
    assert q4.q4_get_device_status() == q4.Q4_OK
    check_guard(raw, M * N, ct, f"M={M} K={K} N={N} {adt}->{cdt} {entry}")


# three launches (T = 1; I = 100 and H = 520 not whole groups of 8 blocks),
# and the persistent form from 4 tokens with H = 504 and I = 252 ragged
# inside their 512-column tiles, and a DeepSeek-like slot count
@pytest.mark.parametrize("T,topk,E,H,I", [(1, 2, 3, 250, 96), (5, 6, 8, 520, 100),
                                         (5, 3, 6, 504, 252), (4, 6, 16, 1024, 512)])
def test_moe_writes_exactly_its_output(T, topk, E, H, I):
    Wg, Wu, Wd = si.moe_weights(E, H, I, seed=T)
    x = si.activations_bf16(T, H, seed=T)
    idx, w = si.routing(T, E, topk, seed=T)
    raw, out = guarded(T * H, torch.float32)
    q4.q4_moe_experts_ex(out.view(T, H), to_dev(x), to_dev(Wg), to_dev(Wu), to_dev(Wd),
                         to_dev(idx), to_dev(w), T, topk, E, H, I)
    torch.cuda.synchronize()
    assert q4.q4_get_device_status() == q4.Q4_OK
    check_guard(raw, T * H, torch.float32, f"moe T={T} H={H}")
