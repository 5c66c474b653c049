"""Seeded synthetic inputs for the Q4_0 dequant-matmul path.

This module is shared by the oracle side and the CUDA side: it only draws
numbers and lays them out in the block format the path consumes.  It holds
none of the path's arithmetic (no dequantisation, no products, no sums).

Recipe (the workloads of the C++ DeepSeek engine page, §2.2-§3.4, and the
DeepSeek-V2 routed-expert shape of the KTransformers page, «优化三»):

* Q4_0 weights for a K x N matrix: K rows, each of nb = ceil(N/32) blocks of
  18 bytes {fp16 d little-endian, uint8 qs[16]}.  Nibbles q are uniform in
  {0..15}; d = fp16_rn(uniform[0.001, 0.01]).  Nibbles of padding columns
  (j >= N in the last block of a row) are written as q = 8, the code whose
  value is exactly zero.
* Activations: fp32 N(0,1); bf16 activations are those fp32 draws rounded to
  bf16 (round to nearest, ties to even), returned as raw uint16 bits.
* Routing for the routed experts: logits N(0,1) of shape [T, E] in fp32,
  softmax with the maximum subtracted first, top-k by descending probability
  with ties to the lower expert index, weights renormalised over the k picks.
  These are inputs of the expert path, not part of it.

Every draw comes from numpy's PCG64 seeded with (seed, stream), so two calls
with the same arguments return identical arrays.
"""

from __future__ import annotations

import numpy as np

BLOCK = 32          # weights per block_q4_0
BLOCK_BYTES = 18    # 2 bytes fp16 scale + 16 bytes of nibbles


def rng(seed: int, stream: int) -> np.random.Generator:
    return np.random.Generator(np.random.PCG64(np.random.SeedSequence([int(seed), int(stream)])))


def nblocks(N: int) -> int:
    return (int(N) + BLOCK - 1) // BLOCK


def q4_weights(K: int, N: int, seed: int = 0, stream: int = 0,
               d_lo: float = 0.001, d_hi: float = 0.01) -> np.ndarray:
    """Q4_0 blocks of a K x N matrix as uint8 [K, nb*18] (row k = nb blocks)."""
    nb = nblocks(N)
    g = rng(seed, stream)
    out = np.empty((K, nb, BLOCK_BYTES), dtype=np.uint8)
    d = g.uniform(d_lo, d_hi, size=(K, nb)).astype(np.float16)
    out[:, :, 0:2] = d.view(np.uint8).reshape(K, nb, 2)
    out[:, :, 2:] = g.integers(0, 256, size=(K, nb, 16), dtype=np.uint8)
    pad = nb * BLOCK - N
    if pad:
        _fill_padding(out, N, 8)
    return out.reshape(K, nb * BLOCK_BYTES)


Q8_BLOCK_BYTES = 34


def q8_weights(K: int, N: int, seed: int = 0, stream: int = 0,
               d_lo: float = 0.001, d_hi: float = 0.01) -> np.ndarray:
    """Q8_0 blocks of a K x N matrix as uint8 [K, nb*34]: per block an fp16
    scale drawn as for Q4_0 and 32 uniform random bytes (int8 codes); padding
    codes are 0."""
    nb = nblocks(N)
    g = rng(seed, stream)
    out = np.empty((K, nb, Q8_BLOCK_BYTES), dtype=np.uint8)
    d = g.uniform(d_lo, d_hi, size=(K, nb)).astype(np.float16)
    out[:, :, 0:2] = d.view(np.uint8).reshape(K, nb, 2)
    out[:, :, 2:] = g.integers(0, 256, size=(K, nb, BLOCK), dtype=np.uint8)
    first = N - (nb - 1) * BLOCK
    out[:, nb - 1, 2 + first:] = 0
    return out.reshape(K, nb * Q8_BLOCK_BYTES)


def _fill_padding(blocks: np.ndarray, N: int, q: int) -> None:
    """Write nibble value q into every padding column of the last block."""
    nb = blocks.shape[1]
    first = N - (nb - 1) * BLOCK          # real columns in the last block
    last = blocks[:, nb - 1, 2:]
    for l in range(first, BLOCK):
        byte = l // 2
        if l % 2 == 0:
            last[:, byte] = (last[:, byte] & 0xF0) | q
        else:
            last[:, byte] = (last[:, byte] & 0x0F) | (q << 4)


def randomise_padding(B: np.ndarray, K: int, N: int, seed: int, stream: int) -> np.ndarray:
    """Copy of B whose padding nibbles hold random codes (a padding-invariance input)."""
    nb = nblocks(N)
    out = B.reshape(K, nb, BLOCK_BYTES).copy()
    first = N - (nb - 1) * BLOCK
    g = rng(seed, stream)
    vals = g.integers(0, 16, size=(K, BLOCK - first), dtype=np.uint8)
    last = out[:, nb - 1, 2:]
    for i, l in enumerate(range(first, BLOCK)):
        byte = l // 2
        if l % 2 == 0:
            last[:, byte] = (last[:, byte] & 0xF0) | vals[:, i]
        else:
            last[:, byte] = (last[:, byte] & 0x0F) | (vals[:, i] << 4)
    return out.reshape(K, nb * BLOCK_BYTES)


def f32_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """Round fp32 to bf16 (nearest, ties to even); NaN stays a quiet NaN."""
    u = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32).astype(np.uint64)
    r = ((u + 0x7FFF + ((u >> 16) & 1)) >> 16).astype(np.uint16)
    nan = np.isnan(x)
    if nan.any():
        r[nan] = 0x7FC0
    return r


def activations_f32(M: int, K: int, seed: int = 0, stream: int = 1) -> np.ndarray:
    return rng(seed, stream).standard_normal(size=(M, K), dtype=np.float32)


def activations_bf16(M: int, K: int, seed: int = 0, stream: int = 1) -> np.ndarray:
    """bf16 N(0,1) activations as raw uint16 bits [M, K]."""
    return f32_to_bf16_bits(activations_f32(M, K, seed, stream))


def router_logits(T: int, E: int, seed: int = 0, stream: int = 2) -> np.ndarray:
    """Seeded N(0,1) router logits, fp32 [T, E]."""
    return rng(seed, stream).standard_normal(size=(T, E), dtype=np.float32)


def routing(T: int, E: int, topk: int, seed: int = 0, stream: int = 2):
    """(topk_idx int32 [T, topk], topk_w fp32 [T, topk]) from seeded N(0,1) logits:
    input data for the expert path (the gate itself is checked against the
    oracle's router)."""
    logits = router_logits(T, E, seed, stream)
    m = logits.max(axis=1, keepdims=True)
    e = np.exp(logits - m, dtype=np.float32)
    p = (e / e.sum(axis=1, keepdims=True, dtype=np.float32)).astype(np.float32)
    # descending probability, ties to the lower expert index (stable sort of -p)
    order = np.argsort(-p, axis=1, kind="stable")[:, :topk]
    idx = order.astype(np.int32)
    w = np.take_along_axis(p, order, axis=1)
    w = (w / w.sum(axis=1, keepdims=True, dtype=np.float32)).astype(np.float32)
    return idx, w


def moe_weights(E: int, H: int, I: int, seed: int = 0):
    """Per-expert Q4_0 weights: W_gate, W_up [E, H, nb(I)*18], W_down [E, I, nb(H)*18]."""
    wg = np.stack([q4_weights(H, I, seed, 1000 + e) for e in range(E)])
    wu = np.stack([q4_weights(H, I, seed, 2000 + e) for e in range(E)])
    wd = np.stack([q4_weights(I, H, seed, 3000 + e) for e in range(E)])
    return wg, wu, wd


# The 7B-like decode sweep: 32 layers of (K, N) shapes, one token.
SWEEP_LAYER = [(4096, 4096)] * 4 + [(4096, 11008)] * 2 + [(11008, 4096)]
SWEEP_LAYERS = 32


def sweep_shapes(layers: int = SWEEP_LAYERS):
    return [s for _ in range(layers) for s in SWEEP_LAYER]
