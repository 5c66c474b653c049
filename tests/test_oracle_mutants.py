"""The oracle's pins catch plausible mistakes.

Each case plants one mistake in a copy of the oracle's C source (on the CPU),
builds it, routes the oracle module to the mutant and runs the pin battery:
at least one pin must fail.  The real oracle is restored afterwards.
"""

import os
import subprocess

import numpy as np
import pytest

import oracle
import test_oracle_pins as pins
import test_oracle_q8_pins as q8pins

MUTANTS = {
    "nibble order swapped": ("(packed & 0x0F) : (packed >> 4)", "(packed >> 4) : (packed & 0x0F)"),
    "scale bytes big-endian": ("blk[0] | (blk[1] << 8)", "blk[1] | (blk[0] << 8)"),
    "offset 8 dropped in matmul": ("double p = av * (double)(q - 8) * d;", "double p = av * (double)(q) * d;"),
    "offset 8 dropped in dequant": ("return (double)(q - 8) * block_scale(blk);", "return (double)(q - 7) * block_scale(blk);"),
    "fp16 exponent bias off by one": ("e - 25);   /* (1 + f/1024)", "e - 24);   /* (1 + f/1024)"),
    "fp16 subnormal scale": ("v = ldexp((double)f, -24);", "v = ldexp((double)f, -25);"),
    "row stride wrong": ("const uint8_t *row = B + k * nb * QO_BLOCK_BYTES;\n        for (int64_t b = 0; b < nb; b++) {\n            const uint8_t *blk = row + b * QO_BLOCK_BYTES;\n            double d = block_scale(blk);\n            for (int l = 0; l < QO_BLOCK; l++) {\n                int64_t j = b * QO_BLOCK + l;\n                if (j >= N)\n                    break;          /* padding column: never stored */",
                         "const uint8_t *row = B + k * nb * QO_BLOCK_BYTES;\n        for (int64_t b = 0; b < nb; b++) {\n            const uint8_t *blk = row + ((b + 1) % nb) * QO_BLOCK_BYTES;\n            double d = block_scale(blk);\n            for (int l = 0; l < QO_BLOCK; l++) {\n                int64_t j = b * QO_BLOCK + l;\n                if (j >= N)\n                    break;          /* padding column: never stored */"),
    "operand transposed": ("a[k] = act_at(A, a_dtype, i * K + k);", "a[k] = act_at(A, a_dtype, k * M + i);"),
    "C accumulated, not zeroed": ("        c[j] = 0.0;\n        if (s)\n            s[j] = 0.0;", "        if (s)\n            s[j] = 0.0;"),
    "sigmoid sign": ("return 1.0 / (1.0 + exp(-g));", "return 1.0 / (1.0 + exp(g));"),
    "routing weight dropped": ("out[t * H + j] += wk * y[j];", "out[t * H + j] += y[j];"),
    "up projection dropped": ("h[i] = silu * u[i];", "h[i] = silu;"),
    "bf16 ties away from zero": ("(diff == 0.5 && fmod(fl, 2.0) != 0.0))\n        r = fl + 1.0;\n    double v = ldexp(r, (int)quantum_exp);",
                                 "(diff == 0.5))\n        r = fl + 1.0;\n    double v = ldexp(r, (int)quantum_exp);"),
    "router ties to the higher index": ("if (!taken[e] && (best < 0 || p[e] > p[best]))", "if (!taken[e] && (best < 0 || p[e] >= p[best]))"),
    "router weights not renormalised": ("            w[t * topk + k] /= wsum;", "            w[t * topk + k] /= 1.0;"),
    "router max not subtracted": ("            p[e] = exp((double)l[e] - mx);", "            p[e] = exp((double)l[e]);"),
    "block shared term dropped": ("        out[i] += so[i];", "        out[i] += 0.0 * so[i];"),
    "block shared weight doubled": ("        sw[t] = 1.0;", "        sw[t] = 2.0;"),
    "encoder truncates instead of rounding": ("                    t = t + 8.5f;", "                    t = t + 8.0f;"),
    "encoder takes the largest value, not magnitude": ("                if (amax < fabsf(v)) {\n                    amax = fabsf(v);", "                if (amax < v) {\n                    amax = v;"),
    "encoder padding code 0": ("                int q = 8;\n                if (l < n) {", "                int q = 0;\n                if (l < n) {"),
    "fp16 ties away from zero": ("    if (diff > 0.5 || (diff == 0.5 && fmod(fl, 2.0) != 0.0))\n        r = fl + 1.0;\n    double v = ldexp(r, quantum_exp);", "    if (diff >= 0.5)\n        r = fl + 1.0;\n    double v = ldexp(r, quantum_exp);"),
    "router picks the smallest": ("if (!taken[e] && (best < 0 || p[e] > p[best]))", "if (!taken[e] && (best < 0 || p[e] < p[best]))"),
    "q8 codes read unsigned": ("    if (q >= 128)\n        q -= 256;                          /* two's complement */", "    (void)0;"),
    "q8 codes offset by one byte": ("    int q = (int)blk[2 + j % QO_BLOCK];", "    int q = (int)blk[1 + j % QO_BLOCK];"),
    "q8 blocks 18 bytes apart": ("    const uint8_t *blk = B + (k * nb + j / QO_BLOCK) * QO_Q8_BYTES;", "    const uint8_t *blk = B + (k * nb + j / QO_BLOCK) * QO_BLOCK_BYTES;"),
    "silu without its g factor": ("double silu = g[i] * sgm;", "double silu = sgm;"),
    "every token reads row 0 of x": ("xt[i] = act_at(x, x_dtype, t * H + i);", "xt[i] = act_at(x, x_dtype, i);"),
    "bf16 exponent bias off by one": ("v = ldexp((double)(128 + f), e - 134);", "v = ldexp((double)(128 + f), e - 133);"),
    "q8 activation row stride": ("            double av = act_at(A, a_dtype, i * K + k);", "            double av = act_at(A, a_dtype, i + k);"),
}

BATTERY = [
    lambda: pins.test_dequant_hand_built_blocks(oracle),
    lambda: pins.test_dequant_all_nibbles_both_positions(oracle),
    lambda: pins.test_fp16_decode_all_codes(oracle),
    lambda: pins.test_bf16_encode_matches_torch(oracle),
    pins.test_layout_one_hot,
    pins.test_zero_cases,
    lambda: pins.test_matmul_exact_rational(2, 3, 64),
    lambda: pins.test_matmul_exact_rational(3, 17, 40),
    pins.test_fused_equals_textbook,
    pins.test_moe_closed_form,
    pins.test_moe_closed_form_two_tokens,
    lambda: pins.test_silu_closed_forms(oracle),
    pins.test_bf16_tiles_hand_rounded,
    pins.test_bf16_tiles_equal_exact_product_when_representable,
    pins.test_bf16_tiles_within_rounding_bound,
    pins.test_gate_closed_forms,
    pins.test_gate_ties_go_to_the_lower_index,
    pins.test_gate_matches_stable_sort,
    pins.test_gate_large_logits_stay_finite,
    pins.test_block_shared_term_is_the_shared_expert,
    pins.test_block_identical_experts_collapse,
    pins.test_block_expert_relabelling,
    lambda: pins.test_fp16_encode_matches_numpy(oracle),
    pins.test_quantize_closed_forms,
    pins.test_quantize_matches_fp32_restatement,
    pins.test_quantize_round_trip_bound,
    q8pins.test_hand_written_blocks,
    lambda: q8pins.test_equals_pinned_q4_on_reencoded_weights(2, 64, 96),
    q8pins.test_layout_one_hot,
    lambda: q8pins.test_exact_rational(2, 5, 40),
    q8pins.test_padding_and_linearity,
]


def _build_mutant(tmp_path, name, old, new):
    with open(os.path.join(os.path.dirname(oracle.__file__), "q4_oracle.c")) as f:
        src = f.read()
    assert src.count(old) == 1, f"mutation site for '{name}' not unique"
    path = tmp_path / "mut.c"
    path.write_text(src.replace(old, new))
    so = tmp_path / "libmut.so"
    subprocess.run(["gcc", "-std=c99", "-O1", "-fPIC", "-shared", str(path), "-o", str(so), "-lm"],
                   check=True)
    return str(so)


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_pins_catch_mutant(name, tmp_path):
    old, new = MUTANTS[name]
    lib = oracle.bind(_build_mutant(tmp_path, name, old, new))
    oracle.use(lib)
    try:
        failed = []
        for check in BATTERY:
            try:
                check()
            except (AssertionError, ValueError, ZeroDivisionError, OverflowError):
                failed.append(check)
        assert failed, f"no pin caught the mutant '{name}'"
    finally:
        oracle.use(None)


# Mistakes in the bf16-tile product (a Python composition of oracle steps):
# each replaces the tile dequantisation and must fail a bf16-tile pin.
def _tiles_truncated(B, K, N):
    W = oracle.dequant_f32(B, K, N)
    return (W.view(np.uint32) >> 16).astype(np.uint16)


def _tiles_ties_up(B, K, N):
    W = oracle.dequant_f32(B, K, N).view(np.uint32).astype(np.uint64)
    return ((W + 0x8000) >> 16).astype(np.uint16)


@pytest.mark.parametrize("mutant", [_tiles_truncated, _tiles_ties_up])
def test_bf16_tile_pins_catch_mutant(mutant, monkeypatch):
    monkeypatch.setattr(oracle, "dequant_bf16", mutant)
    tiles = [pins.test_bf16_tiles_hand_rounded,
             pins.test_bf16_tiles_equal_exact_product_when_representable,
             pins.test_bf16_tiles_within_rounding_bound]
    failed = 0
    for t in tiles:
        try:
            t()
        except AssertionError:
            failed += 1
    assert failed > 0


def test_bf16_tile_pins_catch_unrounded_tiles(monkeypatch):
    """Tiles that keep the exact fp32 weight (no bf16 rounding at all)."""
    real = oracle.matmul_bf16_tiles

    def unrounded(A, B, M, N, K):
        A = np.ascontiguousarray(A)
        A64 = ((A.astype(np.uint32) << 16).view(np.float32) if A.dtype == np.uint16
               else A.astype(np.float32)).astype(np.float64).reshape(M, K)
        W = oracle.dequant_f32(B, K, N).astype(np.float64)
        return A64 @ W, np.abs(A64) @ np.abs(W)

    monkeypatch.setattr(oracle, "matmul_bf16_tiles", unrounded)
    with pytest.raises(AssertionError):
        pins.test_bf16_tiles_hand_rounded()
    monkeypatch.setattr(oracle, "matmul_bf16_tiles", real)
