"""Helpers of the GPU parity tests: device transfer and the matmul tolerance."""

import numpy as np
import pytest

torch = pytest.importorskip("torch")


def device():
    return torch.device("cuda:0")


def to_dev(a):
    a = np.ascontiguousarray(a)
    if a.dtype == np.uint16:
        return torch.from_numpy(a.view(np.int16)).to(device()).view(torch.bfloat16)
    return torch.from_numpy(a).to(device())


def to_host64(t):
    return t.detach().float().cpu().numpy().astype(np.float64)


def assert_within_matmul_tol(got, C64, S, what=""):
    """|gpu - oracle| <= 1e-3 * sum_k |a*w| + 1e-6 element by element."""
    err = np.abs(got - C64)
    tol = 1e-3 * S + 1e-6
    bad = ~(err <= tol)
    if bad.any():
        i = np.argwhere(bad)[0]
        raise AssertionError(f"{what}: {bad.sum()} elements out of tolerance, first {tuple(i)}: "
                             f"gpu {got[tuple(i)]!r} oracle {C64[tuple(i)]!r} tol {tol[tuple(i)]!r}")
    return float(np.max(err / tol)) if err.size else 0.0


def f32_bits(a):
    return np.ascontiguousarray(a, dtype=np.float32).view(np.uint32)


def same_f32(a, b):
    """Bit-identical fp32 arrays, any NaN matching any NaN."""
    a = np.asarray(a, np.float32)
    b = np.asarray(b, np.float32)
    na, nb = np.isnan(a), np.isnan(b)
    return bool(np.array_equal(na, nb) and np.array_equal(f32_bits(np.where(na, 0, a)),
                                                          f32_bits(np.where(nb, 0, b))))


def same_bf16(a, b):
    """Bit-identical bf16 codes, any NaN code matching any NaN code (NaN
    payloads are not pinned by the block definition)."""
    a = np.asarray(a, np.uint16)
    b = np.asarray(b, np.uint16)
    na = ((a & 0x7F80) == 0x7F80) & ((a & 0x7F) != 0)
    nb = ((b & 0x7F80) == 0x7F80) & ((b & 0x7F) != 0)
    return bool(np.array_equal(na, nb) and np.array_equal(np.where(na, 0, a), np.where(nb, 0, b)))
