"""The routed experts' workspace on the host (no GPU): q4_moe_workspace_size.

The workspace (KTransformers page «优化三»: the chosen experts' GEMVs, their
intermediate rows kept on the device) is a 64 KB counter header followed by
the rows of the form the call prefers.  The three-launch form needs the
SiLU(g)·u rows h [T·topk, I] and the per-slot down rows y [T·topk, H]; the
persistent form (from 4 tokens, at most 512 slots, whole 256-column block
groups in I and H) needs g, u, h and y and the partial rows of its K slices
(2 KB per unit of work).  A workspace of at least the header plus the
three-launch rows runs the three-launch form.
"""

import pytest

import quantized_weight_q4_gb300 as q4

HEADER = 64 * 1024


def r256(n):
    return -(-n // 256) * 256


def three_launch_rows(T, topk, H, I):
    S = T * topk
    return r256(S * I * 4) + r256(S * H * 4)


@pytest.mark.parametrize("T,topk,E,H,I", [
    (1, 6, 160, 5120, 1536),     # one token
    (3, 6, 160, 5120, 1536),     # below the persistent form's 4 tokens
    (8, 6, 160, 5120, 320),      # I = 320: 10 blocks per row, not whole groups of 8
    (100, 6, 160, 5120, 1536),   # 600 slots, more than 512
])
def test_shapes_the_persistent_form_does_not_take(T, topk, E, H, I):
    assert q4.q4_moe_workspace_size(T, topk, E, H, I) == HEADER + three_launch_rows(T, topk, H, I)


@pytest.mark.parametrize("T,topk,E,H,I", [
    (4, 6, 160, 5120, 1536), (8, 6, 160, 5120, 1536), (32, 6, 160, 5120, 1536),
    (5, 2, 7, 4328, 256), (8, 2, 3, 512, 4608)])
def test_shapes_the_persistent_form_takes(T, topk, E, H, I):
    n = q4.q4_moe_workspace_size(T, topk, E, H, I)
    S = T * topk
    # g, u, h and y, plus at least one 2 KB partial row per gate/up unit
    assert n >= HEADER + 3 * r256(S * I * 4) + r256(S * H * 4) + 2 * S * 2048
    assert n > HEADER + three_launch_rows(T, topk, H, I)


def test_deepseek_v2_32_tokens_layout():
    """192 slots: g, u, h of 192 x 1536 fp32, y of 192 x 5120 fp32, and the
    partial rows of gate/up (2 x 192 slots x 3 column tiles x 2 K slices of
    2560 rows = 2304 units of 2 KB; down takes I = 1536 in one slice)."""
    T, topk, E, H, I = 32, 6, 160, 5120, 1536
    S = T * topk
    want = HEADER + 3 * r256(S * I * 4) + r256(S * H * 4) + 2 * S * 3 * 2 * 2048
    assert q4.q4_moe_workspace_size(T, topk, E, H, I) == want


def test_sizes_grow_with_tokens():
    sizes = [q4.q4_moe_workspace_size(T, 6, 160, 5120, 1536) for T in (1, 2, 4, 8, 16, 32)]
    assert sizes == sorted(sizes) and len(set(sizes)) == len(sizes)


def test_argument_errors_give_zero():
    assert q4.q4_moe_workspace_size(0, 6, 160, 5120, 1536) == 0
    assert q4.q4_moe_workspace_size(1, 0, 160, 5120, 1536) == 0
    assert q4.q4_moe_workspace_size(1, 6, 160, 0, 1536) == 0
