"""The CPU baseline of the benchmark: the engine page's fused fp32 Q4_0 loop
with OpenMP over column blocks (``q4_cpu.c``), built with the host C compiler
into ``cpu_baseline/_build/``.  Benchmark infrastructure: bench.py times it
next to the GPU path; nothing in the package or the oracle uses it."""

from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "q4_cpu.c")
_LIB = os.path.join(_HERE, "_build", "libq4_cpu.so")
_lib = None


def build() -> str:
    os.makedirs(os.path.dirname(_LIB), exist_ok=True)
    if os.path.exists(_LIB) and os.path.getmtime(_LIB) >= os.path.getmtime(_SRC):
        return _LIB
    tmp = _LIB + f".tmp{os.getpid()}"
    subprocess.run(["gcc", "-std=c99", "-O3", "-fopenmp", "-fPIC", "-shared", _SRC, "-o", tmp,
                    "-lm"], check=True)
    os.replace(tmp, _LIB)
    return _LIB


def lib() -> ctypes.CDLL:
    global _lib
    if _lib is None:
        L = ctypes.CDLL(build())
        L.q4cpu_matmul.argtypes = [ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p,
                                   ctypes.c_int64, ctypes.c_int64, ctypes.c_int64, ctypes.c_int]
        L.q4cpu_matmul.restype = ctypes.c_int
        _lib = L
    return _lib


def physical_cores() -> int:
    """Physical cores of the host (one thread each, as the page advises)."""
    try:
        out = subprocess.run(["lscpu", "-p=CORE,SOCKET"], capture_output=True, text=True,
                             check=True).stdout
        cores = {tuple(l.split(",")) for l in out.splitlines() if l and not l.startswith("#")}
        if cores:
            return len(cores)
    except (OSError, subprocess.CalledProcessError):
        pass
    return os.cpu_count() or 1


def matmul(A: np.ndarray, B: np.ndarray, M: int, N: int, K: int, threads: int) -> np.ndarray:
    A = np.ascontiguousarray(A, dtype=np.float32)
    B = np.ascontiguousarray(B, dtype=np.uint8)
    C = np.empty((M, N), dtype=np.float32)
    rc = lib().q4cpu_matmul(A.ctypes.data, B.ctypes.data, C.ctypes.data, M, N, K, threads)
    if rc != 0:
        raise ValueError("q4cpu_matmul: bad arguments")
    return C
