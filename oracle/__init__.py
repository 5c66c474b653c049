"""ctypes access to the fp64 CPU oracle of the Q4_0 dequant-matmul.

TEST INFRASTRUCTURE.  Only the tests, ``__graft_entry__.smoke()`` and the
CPU-baseline leg of ``bench.py`` may import this package.  It never imports
the CUDA package and the CUDA package never imports it.

``build()`` compiles ``q4_oracle.c`` with the host C compiler into
``oracle/_build/`` (plain C99, portable to x86-64 and aarch64 hosts).
"""

from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "q4_oracle.c")
_OUT_DIR = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_OUT_DIR, "liboracle_q4.so")
_lock = threading.Lock()
_lib = None

_DT = {"f32": 0, "bf16": 1}


def build(force: bool = False) -> str:
    """Compile the oracle if its library is missing or older than its source."""
    os.makedirs(_OUT_DIR, exist_ok=True)
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)):
        return _LIB_PATH
    tmp = _LIB_PATH + f".tmp{os.getpid()}"
    cmd = ["gcc", "-std=c99", "-O2", "-fPIC", "-shared", "-Wall", _SRC, "-o", tmp, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def bind(path: str) -> ctypes.CDLL:
    """Load an oracle library from ``path`` and declare its signatures."""
    L = ctypes.CDLL(path)
    c_i64, vp = ctypes.c_int64, ctypes.c_void_p
    L.q4o_fp16_to_f64.argtypes = [ctypes.c_uint16]
    L.q4o_fp16_to_f64.restype = ctypes.c_double
    L.q4o_bf16_to_f64.argtypes = [ctypes.c_uint16]
    L.q4o_bf16_to_f64.restype = ctypes.c_double
    L.q4o_f64_to_bf16.argtypes = [ctypes.c_double]
    L.q4o_f64_to_bf16.restype = ctypes.c_uint16
    L.q4o_silu.argtypes = [ctypes.c_double]
    L.q4o_silu.restype = ctypes.c_double
    L.q4o_dequant_f32.argtypes = [vp, c_i64, c_i64, vp]
    L.q4o_dequant_bf16.argtypes = [vp, c_i64, c_i64, vp]
    L.q4o_matmul.argtypes = [vp, ctypes.c_int, vp, c_i64, c_i64, c_i64, vp, vp]
    L.q4o_matmul_naive.argtypes = [vp, ctypes.c_int, vp, c_i64, c_i64, c_i64, vp]
    L.q4o_moe_gate.argtypes = [vp, c_i64, c_i64, c_i64, vp, vp]
    L.q4o_f64_to_fp16.argtypes = [ctypes.c_double]
    L.q4o_f64_to_fp16.restype = ctypes.c_uint16
    L.q4o_quantize.argtypes = [vp, ctypes.c_int, c_i64, c_i64, vp]
    L.q4o_q8_dequant_f32.argtypes = [vp, c_i64, c_i64, vp]
    L.q4o_q8_matmul.argtypes = [vp, ctypes.c_int, vp, c_i64, c_i64, c_i64, vp, vp]
    L.q4o_moe_block.argtypes = [vp, ctypes.c_int, vp, vp, vp, vp, c_i64, c_i64, c_i64, c_i64, c_i64,
                                vp, vp, vp, c_i64, vp, vp, vp, vp]
    L.q4o_moe.argtypes = [vp, ctypes.c_int, vp, vp, vp, vp, vp,
                          c_i64, c_i64, c_i64, c_i64, c_i64,
                          vp, vp, vp, vp, vp]
    return L


def lib() -> ctypes.CDLL:
    """The oracle library built from ``q4_oracle.c`` (or one set by ``use``)."""
    global _lib
    with _lock:
        if _lib is None:
            _lib = bind(build())
        return _lib


def use(L) -> None:
    """Route this module's functions to library ``L`` (None: the built one)."""
    global _lib
    with _lock:
        _lib = L


def _p(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def _act(A: np.ndarray):
    """(contiguous array, dtype code): fp32 values or bf16 raw uint16 bits."""
    A = np.ascontiguousarray(A)
    if A.dtype == np.float32:
        return A, _DT["f32"]
    if A.dtype == np.uint16:
        return A, _DT["bf16"]
    raise TypeError(f"activations must be float32 or uint16 bf16 bits, not {A.dtype}")


def fp16_to_f64(h: int) -> float:
    return lib().q4o_fp16_to_f64(h)


def bf16_to_f64(h: int) -> float:
    return lib().q4o_bf16_to_f64(h)


def f64_to_bf16(x: float) -> int:
    return lib().q4o_f64_to_bf16(x)


def f64_to_fp16(x: float) -> int:
    return lib().q4o_f64_to_fp16(x)


def quantize(W: np.ndarray, K: int, N: int) -> np.ndarray:
    """Q4_0 blocks [K, nb*18] of W (fp32, or bf16 bits as uint16) by the
    oracle's encoder."""
    W, dt = _act(W)
    B = np.empty((K, ((N + 31) // 32) * 18), dtype=np.uint8)
    lib().q4o_quantize(_p(W), dt, K, N, _p(B))
    return B


def silu(g: float) -> float:
    return lib().q4o_silu(g)


def dequant_f32(B: np.ndarray, K: int, N: int) -> np.ndarray:
    B = np.ascontiguousarray(B, dtype=np.uint8)
    W = np.empty((K, N), dtype=np.float32)
    lib().q4o_dequant_f32(_p(B), K, N, _p(W))
    return W


def dequant_bf16(B: np.ndarray, K: int, N: int) -> np.ndarray:
    B = np.ascontiguousarray(B, dtype=np.uint8)
    W = np.empty((K, N), dtype=np.uint16)
    lib().q4o_dequant_bf16(_p(B), K, N, _p(W))
    return W


def matmul(A: np.ndarray, B: np.ndarray, M: int, N: int, K: int, with_abs: bool = True):
    """(C64 [M,N], S [M,N] or None): fp64 product and sum_k |a*w|."""
    A, dt = _act(A)
    B = np.ascontiguousarray(B, dtype=np.uint8)
    C = np.empty((M, N), dtype=np.float64)
    S = np.empty((M, N), dtype=np.float64) if with_abs else None
    lib().q4o_matmul(_p(A), dt, _p(B), M, N, K, _p(C), _p(S))
    return C, S


def q8_dequant_f32(B: np.ndarray, K: int, N: int) -> np.ndarray:
    """Q8_0 blocks (34 bytes: fp16 d, int8 q[32]) -> W [K, N] fp32 = q * d."""
    B = np.ascontiguousarray(B, dtype=np.uint8)
    W = np.empty((K, N), dtype=np.float32)
    lib().q4o_q8_dequant_f32(_p(B), K, N, _p(W))
    return W


def q8_matmul(A: np.ndarray, B: np.ndarray, M: int, N: int, K: int, with_abs: bool = True):
    """(C64 [M,N], S [M,N] or None) for Q8_0 weights."""
    A, dt = _act(A)
    B = np.ascontiguousarray(B, dtype=np.uint8)
    C = np.empty((M, N), dtype=np.float64)
    S = np.empty((M, N), dtype=np.float64) if with_abs else None
    lib().q4o_q8_matmul(_p(A), dt, _p(B), M, N, K, _p(C), _p(S))
    return C, S


def matmul_bf16_tiles(A: np.ndarray, B: np.ndarray, M: int, N: int, K: int):
    """(C64 [M,N], S [M,N]): A . bf16_rn(W) in fp64, with S = sum_k |a * bf16_rn(w)|.

    The product of the tensor-core prefill path, which batches a prompt's
    tokens into one matmul (C++ DeepSeek engine page, §5.2) and dequantises
    each weight to a bf16 tile element before the multiply.  Reading: the
    pages fix no tile precision; bf16 is the tensor cores' input type, and
    each weight is rounded once, to nearest even, from its exact value.
    Steps: the C oracle's bf16 dequantisation, the bf16 bit patterns widened
    to fp64 (16 zero bits appended to make the fp32 pattern), then one fp64
    matmul (a library primitive).  Every product is exact in fp64 (8-bit
    bf16 times an 8-bit bf16 or 24-bit fp32 activation).
    """
    A = np.ascontiguousarray(A)
    if A.dtype == np.uint16:
        A64 = (A.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    else:
        A64 = A.astype(np.float32).astype(np.float64)
    Wb = dequant_bf16(B, K, N)
    W64 = (Wb.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    A64 = A64.reshape(M, K)
    return A64 @ W64, np.abs(A64) @ np.abs(W64)


def matmul_naive(A: np.ndarray, B: np.ndarray, M: int, N: int, K: int) -> np.ndarray:
    A, dt = _act(A)
    B = np.ascontiguousarray(B, dtype=np.uint8)
    C = np.empty((M, N), dtype=np.float64)
    lib().q4o_matmul_naive(_p(A), dt, _p(B), M, N, K, _p(C))
    return C


def moe_gate(logits, T: int, E: int, topk: int):
    """(topk_idx int32 [T, topk], topk_w fp64 [T, topk]): softmax of each
    token's fp32 logits (max subtracted), the topk largest in descending order
    (ties: lower index first), renormalised; fp64."""
    logits = np.ascontiguousarray(logits, dtype=np.float32)
    idx = np.empty((T, topk), dtype=np.int32)
    w = np.empty((T, topk), dtype=np.float64)
    lib().q4o_moe_gate(_p(logits), T, E, topk, _p(idx), _p(w))
    return idx, w


def moe_block(x, logits, Wg, Wu, Wd, T, topk, E, H, I, Sg=None, Su=None, Sd=None, Is=0):
    """(out [T,H], tol [T,H], idx [T,topk], w [T,topk]) of one MoE block:
    router, routed experts, shared expert (Is > 0); fp64."""
    x, dt = _act(x)
    logits = np.ascontiguousarray(logits, dtype=np.float32)
    Wg, Wu, Wd = (np.ascontiguousarray(a, dtype=np.uint8) for a in (Wg, Wu, Wd))
    sh = [np.ascontiguousarray(a, dtype=np.uint8) if a is not None else None for a in (Sg, Su, Sd)]
    out = np.empty((T, H), np.float64)
    tol = np.empty((T, H), np.float64)
    idx = np.empty((T, topk), np.int32)
    w = np.empty((T, topk), np.float64)
    lib().q4o_moe_block(_p(x), dt, _p(logits), _p(Wg), _p(Wu), _p(Wd), T, topk, E, H, I,
                        _p(sh[0]), _p(sh[1]), _p(sh[2]), Is, _p(out), _p(tol), _p(idx), _p(w))
    return out, tol, idx, w


def moe(x, Wg, Wu, Wd, idx, w, T, topk, E, H, I, stages: bool = False):
    """(out [T,H], tol [T,H], (g, u, h) [T*topk, I] or None), all fp64."""
    x, dt = _act(x)
    Wg = np.ascontiguousarray(Wg, dtype=np.uint8)
    Wu = np.ascontiguousarray(Wu, dtype=np.uint8)
    Wd = np.ascontiguousarray(Wd, dtype=np.uint8)
    idx = np.ascontiguousarray(idx, dtype=np.int32)
    w = np.ascontiguousarray(w, dtype=np.float32)
    out = np.empty((T, H), dtype=np.float64)
    tol = np.empty((T, H), dtype=np.float64)
    g = u = h = None
    if stages:
        g = np.empty((T * topk, I), dtype=np.float64)
        u = np.empty_like(g)
        h = np.empty_like(g)
    lib().q4o_moe(_p(x), dt, _p(Wg), _p(Wu), _p(Wd), _p(idx), _p(w),
                  T, topk, E, H, I, _p(out), _p(tol), _p(g), _p(u), _p(h))
    return out, tol, ((g, u, h) if stages else None)

