"""GB300 (sm_103a) Q4_0 weight-only dequant-matmul: the Python binding.

A thin ctypes layer over the C ABI declared in ``include/q4.h``.  Every
function marshals arguments only (device pointers, sizes, the current torch
stream) and calls the library; all arithmetic runs in the CUDA kernels.
PyTorch provides device memory and streams.

If the compiled library is missing, importing this package raises: there is
no CPU fallback.
"""

from __future__ import annotations

import ctypes
import os
import threading

from . import _build

Q4_OK = 0
Q4_ERR_ARG = -1
Q4_ERR_DTYPE = -2
Q4_ERR_ALIGN = -3
Q4_ERR_CUDA = -4
Q4_ERR_WORKSPACE = -5
Q4_ERR_SHAPE = -6
Q4_ERR_DEVICE = -7
Q4_DEVERR_INDEX = 0x1
Q4_DEVERR_TIMEOUT = 0x2
Q4_F32 = 0
Q4_BF16 = 1
Q4_LAYOUT_BLOCKS = 0
Q4_LAYOUT_PLANAR = 1
Q4_LAYOUT_Q8_0 = 2

_lock = threading.Lock()
_lib = None

_vp = ctypes.c_void_p
_i64 = ctypes.c_int64
_sz = ctypes.c_size_t
_int = ctypes.c_int


class SeqOp(ctypes.Structure):
    """q4_seq_op of include/q4.h: one matmul of a host-streamed sequence."""
    _fields_ = [("C", ctypes.c_void_p), ("A", ctypes.c_void_p), ("B", ctypes.c_void_p),
                ("M", ctypes.c_int64), ("N", ctypes.c_int64), ("K", ctypes.c_int64),
                ("a_dtype", ctypes.c_int), ("c_dtype", ctypes.c_int)]


class GemvOp(ctypes.Structure):
    """q4_gemv_op of include/q4.h: one M = 1 GEMV of a decode sequence."""
    _fields_ = [("C", ctypes.c_void_p), ("A", ctypes.c_void_p), ("B", ctypes.c_void_p),
                ("N", ctypes.c_int64), ("K", ctypes.c_int64),
                ("a_dtype", ctypes.c_int), ("c_dtype", ctypes.c_int),
                ("ndeps", ctypes.c_int), ("deps", ctypes.c_int * 4), ("slice_rows", ctypes.c_int)]


# name -> (restype, argtypes), as declared in include/q4.h
SIGNATURES = {
    "q4_matmul": (_int, [_vp, _vp, _vp, _i64, _i64, _i64]),
    "q4_matmul_ex": (_int, [_vp, _int, _vp, _int, _vp, _int, _i64, _i64, _i64, _vp, _sz, _vp]),
    "q4_matmul_workspace_size": (_sz, [_i64, _i64, _i64]),
    "q4_matmul_bf16_tiles": (_int, [_vp, _int, _vp, _vp, _i64, _i64, _i64, _vp, _sz, _vp]),
    "q4_release_scratch": (_int, []),
    "q4_moe_experts": (_int, [_vp, _vp, _vp, _vp, _vp, _vp, _vp, _i64, _i64, _i64, _i64]),
    "q4_moe_experts_ex": (_int, [_vp, _vp, _int, _vp, _vp, _vp, _vp, _vp,
                                 _i64, _i64, _i64, _i64, _i64, _vp, _sz, _vp]),
    "q4_moe_workspace_size": (_sz, [_i64, _i64, _i64, _i64, _i64]),
    "q4_moe_experts_trace": (_int, [_vp, _vp, _int, _vp, _vp, _vp, _vp, _vp,
                                    _i64, _i64, _i64, _i64, _i64, _vp, _sz,
                                    _vp, _vp, _vp, _vp, _vp]),
    "q4_moe_experts_noalloc": (_int, [_vp, _vp, _int, _vp, _vp, _vp, _vp, _vp,
                                      _i64, _i64, _i64, _i64, _i64, _vp]),
    "q4_moe_static_scratch_bytes": (_sz, []),
    "q4_repack": (_int, [_vp, _vp, _i64, _i64, _vp]),
    "q4_unpack": (_int, [_vp, _vp, _i64, _i64, _vp]),
    "q4_planar_qs_offset": (_sz, [_i64, _i64]),
    "q4_planar_bytes": (_sz, [_i64, _i64]),
    "q4_dequant": (_int, [_vp, _vp, _i64, _i64, _vp]),
    "q4_dequant_bf16": (_int, [_vp, _vp, _i64, _i64, _vp]),
    "q4_quantize": (_int, [_vp, _vp, _int, _i64, _i64, _vp]),
    "q4_moe_gate": (_int, [_vp, _vp, _vp, _i64, _i64, _i64, _vp]),
    "q4_moe_block": (_int, [_vp, _vp, _int, _vp, _vp, _vp, _vp, _i64, _i64, _i64, _i64, _i64,
                            _vp, _vp, _vp, _i64, _vp, _sz, _vp]),
    "q4_moe_block_workspace_size": (_sz, [_i64, _i64, _i64, _i64, _i64, _i64]),
    "q4_selftest_wait": (_int, [_i64, _int, _vp]),
    "q4_prefill_units": (_i64, [_i64, _i64, _i64, _int, _vp, _i64]),
    "q4_host_stream_slot_bytes": (_sz, [ctypes.POINTER(SeqOp), _int]),
    "q4_matmul_host_stream": (_int, [ctypes.POINTER(SeqOp), _int, _vp, _sz, _int, _vp, _vp]),
    "q4_gemv_seq_bytes": (_sz, [ctypes.POINTER(GemvOp), _int]),
    "q4_gemv_seq_create": (_int, [ctypes.POINTER(GemvOp), _int, _vp, _sz,
                                  ctypes.POINTER(ctypes.c_void_p)]),
    "q4_gemv_seq_run": (_int, [_vp, _vp]),
    "q4_gemv_seq_destroy": (None, [_vp]),
    "q4_gemv_seq_grid": (_int, [_vp]),
    "q4_get_device_status": (_int, [_vp]),
    "q4_last_device_flags": (ctypes.c_uint, []),
    "q4_status_str": (ctypes.c_char_p, [_int]),
    "q4_version": (_int, []),
}


class Q4Error(RuntimeError):
    def __init__(self, fn: str, status: int):
        super().__init__(f"{fn} failed: {status} ({status_str(status)})")
        self.status = status


def library_path() -> str:
    return _build.LIB_PATH


def lib() -> ctypes.CDLL:
    """The loaded C library; raises if it has not been built."""
    global _lib
    with _lock:
        if _lib is None:
            path = _build.LIB_PATH
            if not os.path.exists(path):
                raise ImportError(
                    f"{path} is missing: build it with quantized_weight_q4_gb300._build.build() "
                    "(or __graft_entry__.build()); there is no CPU fallback")
            L = ctypes.CDLL(path)
            for name, (res, args) in SIGNATURES.items():
                f = getattr(L, name)
                f.restype = res
                f.argtypes = args
            _lib = L
        return _lib


def status_str(status: int) -> str:
    return lib().q4_status_str(int(status)).decode()


def _check(fn: str, status: int) -> None:
    if status != Q4_OK:
        raise Q4Error(fn, status)


# ------------------------------------------------------------------ helpers
def _ptr(t) -> int | None:
    if t is None:
        return None
    return t.data_ptr()


def _stream(stream) -> int | None:
    """cudaStream_t of a torch stream (default: torch's current stream)."""
    import torch
    if stream is None:
        stream = torch.cuda.current_stream()
    return stream.cuda_stream or None


def _dtype_code(t) -> int:
    import torch
    if t.dtype == torch.float32:
        return Q4_F32
    if t.dtype in (torch.bfloat16, torch.int16, torch.uint16):
        return Q4_BF16
    raise TypeError(f"unsupported dtype {t.dtype}")


def _require_cuda(*ts):
    for t in ts:
        if t is not None and not t.is_cuda:
            raise ValueError("all tensors must be CUDA tensors (there is no CPU path)")
        if t is not None and not t.is_contiguous():
            raise ValueError("all tensors must be contiguous")


# ------------------------------------------------------------------ entry points
def q4_matmul(C, A, B, M: int, N: int, K: int) -> None:
    """C = A . W (fp32 A and C, legacy default stream), as the C entry point."""
    _require_cuda(C, A, B)
    _check("q4_matmul", lib().q4_matmul(_ptr(C), _ptr(A), _ptr(B), M, N, K))


def q4_matmul_ex(C, A, B, M: int, N: int, K: int, workspace=None, stream=None,
                 b_layout: int = Q4_LAYOUT_BLOCKS) -> None:
    _require_cuda(C, A, B, workspace)
    ws_bytes = workspace.numel() * workspace.element_size() if workspace is not None else 0
    _check("q4_matmul_ex", lib().q4_matmul_ex(
        _ptr(C), _dtype_code(C), _ptr(A), _dtype_code(A), _ptr(B), b_layout,
        M, N, K, _ptr(workspace), ws_bytes, _stream(stream)))


def q4_matmul_bf16_tiles(C, A, B, M: int, N: int, K: int, workspace=None, stream=None) -> None:
    """C = A . bf16_rn(W) on the tensor cores (bf16 A), whatever K."""
    _require_cuda(C, A, B, workspace)
    if _dtype_code(A) != Q4_BF16:
        raise TypeError("q4_matmul_bf16_tiles takes bf16 activations")
    ws_bytes = workspace.numel() * workspace.element_size() if workspace is not None else 0
    _check("q4_matmul_bf16_tiles", lib().q4_matmul_bf16_tiles(
        _ptr(C), _dtype_code(C), _ptr(A), _ptr(B), M, N, K, _ptr(workspace), ws_bytes,
        _stream(stream)))


def q4_release_scratch() -> None:
    """Frees the library-owned scratch and workspaces of the current device."""
    _check("q4_release_scratch", lib().q4_release_scratch())


def _seq_ops(ops):
    """ops: list of (C, A, B_host, M, N, K): C and A CUDA tensors, B a pinned CPU tensor."""
    arr = (SeqOp * len(ops))()
    for i, (C, A, B, M, N, K) in enumerate(ops):
        _require_cuda(C, A)
        arr[i] = SeqOp(_ptr(C), _ptr(A), B.data_ptr(), M, N, K, _dtype_code(A), _dtype_code(C))
    return arr


def q4_host_stream_slot_bytes(ops) -> int:
    return lib().q4_host_stream_slot_bytes(_seq_ops(ops), len(ops))


def q4_matmul_host_stream(ops, staging, slots: int, stream=None, copy_stream=None) -> None:
    """Runs ops [(C, A, B_host, M, N, K), ...] in order on `stream`, copying each
    pinned host B into one of `slots` slots of the device buffer `staging` on
    `copy_stream` while earlier matmuls run."""
    _require_cuda(staging)
    arr = _seq_ops(ops)
    nbytes = staging.numel() * staging.element_size()
    _check("q4_matmul_host_stream", lib().q4_matmul_host_stream(
        arr, len(ops), _ptr(staging), nbytes, slots, _stream(stream), _stream(copy_stream)))


def _gemv_ops(ops, slice_rows=0):
    arr = (GemvOp * len(ops))()
    for i, op in enumerate(ops):
        C, A, B, N, K = op[:5]
        deps = list(op[5]) if len(op) > 5 else []
        _require_cuda(C, A, B)
        if len(deps) > 4:
            raise ValueError("at most 4 dependencies per op")
        d = (ctypes.c_int * 4)(*(deps + [0] * (4 - len(deps))))
        arr[i] = GemvOp(_ptr(C), _ptr(A), _ptr(B), N, K, _dtype_code(A), _dtype_code(C),
                        len(deps), d, slice_rows)
    return arr


class GemvSequence:
    """A decode sequence of M = 1 GEMVs run by one persistent launch
    (q4_gemv_seq_*).  ops: list of (C, A, B, N, K) or (C, A, B, N, K, deps),
    CUDA tensors, deps a list of indices of earlier ops whose C must be
    complete before this op reads A.  slice_rows: rows per unit of work for
    every op, a multiple of 64 up to 4096 (0: the library's choice, which
    shortens the units of ops that others wait for and of the sequence's
    last weights).  The tensors are referenced by the
    plan and kept alive with it."""

    def __init__(self, ops, slice_rows: int = 0):
        import torch
        self.ops = list(ops)
        arr = _gemv_ops(self.ops, slice_rows)
        L = lib()
        nbytes = L.q4_gemv_seq_bytes(arr, len(self.ops))
        if nbytes == 0:
            raise Q4Error("q4_gemv_seq_bytes", Q4_ERR_ARG)
        self.buf = torch.empty(nbytes, dtype=torch.uint8, device=self.ops[0][0].device)
        plan = ctypes.c_void_p()
        _check("q4_gemv_seq_create", L.q4_gemv_seq_create(arr, len(self.ops), _ptr(self.buf),
                                                          nbytes, ctypes.byref(plan)))
        self.plan = plan

    def run(self, stream=None) -> None:
        _check("q4_gemv_seq_run", lib().q4_gemv_seq_run(self.plan, _stream(stream)))

    @property
    def grid(self) -> int:
        return lib().q4_gemv_seq_grid(self.plan)

    def __del__(self):
        plan = getattr(self, "plan", None)
        if plan is not None and _lib is not None:
            _lib.q4_gemv_seq_destroy(plan)
            self.plan = None


def q4_matmul_workspace_size(M: int, N: int, K: int) -> int:
    return lib().q4_matmul_workspace_size(M, N, K)


def q4_moe_experts(out, x, W_gate, W_up, W_down, topk_idx, topk_w, T: int, E: int, H: int,
                   I: int) -> None:
    _require_cuda(out, x, W_gate, W_up, W_down, topk_idx, topk_w)
    _check("q4_moe_experts", lib().q4_moe_experts(
        _ptr(out), _ptr(x), _ptr(W_gate), _ptr(W_up), _ptr(W_down), _ptr(topk_idx),
        _ptr(topk_w), T, E, H, I))


def q4_moe_experts_ex(out, x, W_gate, W_up, W_down, topk_idx, topk_w, T: int, topk: int, E: int,
                      H: int, I: int, workspace=None, stream=None) -> None:
    _require_cuda(out, x, W_gate, W_up, W_down, topk_idx, topk_w, workspace)
    ws_bytes = workspace.numel() * workspace.element_size() if workspace is not None else 0
    _check("q4_moe_experts_ex", lib().q4_moe_experts_ex(
        _ptr(out), _ptr(x), _dtype_code(x), _ptr(W_gate), _ptr(W_up), _ptr(W_down),
        _ptr(topk_idx), _ptr(topk_w), T, topk, E, H, I, _ptr(workspace), ws_bytes,
        _stream(stream)))


def q4_moe_experts_trace(out, x, W_gate, W_up, W_down, topk_idx, topk_w, T: int, topk: int,
                         E: int, H: int, I: int, workspace, g, u, h, y, stream=None) -> None:
    """q4_moe_experts_ex that also writes g, u, h [T*topk, I] and y [T*topk, H]."""
    _require_cuda(out, x, W_gate, W_up, W_down, topk_idx, topk_w, workspace, g, u, h, y)
    ws_bytes = workspace.numel() * workspace.element_size()
    _check("q4_moe_experts_trace", lib().q4_moe_experts_trace(
        _ptr(out), _ptr(x), _dtype_code(x), _ptr(W_gate), _ptr(W_up), _ptr(W_down),
        _ptr(topk_idx), _ptr(topk_w), T, topk, E, H, I, _ptr(workspace), ws_bytes,
        _ptr(g), _ptr(u), _ptr(h), _ptr(y), _stream(stream)))


def q4_moe_workspace_size(T: int, topk: int, E: int, H: int, I: int) -> int:
    return lib().q4_moe_workspace_size(T, topk, E, H, I)


def q4_moe_experts_noalloc(out, x, W_gate, W_up, W_down, topk_idx, topk_w, T: int, topk: int,
                           E: int, H: int, I: int, stream=None) -> None:
    """Routed experts with the library's built-in scratch: no device memory
    is allocated, for callers that cannot allocate (see include/q4.h)."""
    _require_cuda(out, x, W_gate, W_up, W_down, topk_idx, topk_w)
    _check("q4_moe_experts_noalloc", lib().q4_moe_experts_noalloc(
        _ptr(out), _ptr(x), _dtype_code(x), _ptr(W_gate), _ptr(W_up), _ptr(W_down),
        _ptr(topk_idx), _ptr(topk_w), T, topk, E, H, I, _stream(stream)))


def q4_quantize(B, W, K: int, N: int, stream=None) -> None:
    """Q4_0 blocks of W (fp32 or bf16) into B (uint8 [K, ceil(N/32)*18])."""
    _require_cuda(B, W)
    _check("q4_quantize", lib().q4_quantize(_ptr(B), _ptr(W), _dtype_code(W), K, N,
                                            _stream(stream)))


def q4_moe_gate(topk_idx, topk_w, logits, T: int, E: int, topk: int, stream=None) -> None:
    _require_cuda(topk_idx, topk_w, logits)
    _check("q4_moe_gate", lib().q4_moe_gate(_ptr(topk_idx), _ptr(topk_w), _ptr(logits), T, E,
                                            topk, _stream(stream)))


def q4_moe_block(out, x, logits, W_gate, W_up, W_down, T: int, topk: int, E: int, H: int, I: int,
                 S_gate=None, S_up=None, S_down=None, Is: int = 0, workspace=None,
                 stream=None) -> None:
    """Router + shared expert + routed experts of one MoE block (include/q4.h)."""
    _require_cuda(out, x, logits, W_gate, W_up, W_down, S_gate, S_up, S_down, workspace)
    ws_bytes = workspace.numel() * workspace.element_size() if workspace is not None else 0
    _check("q4_moe_block", lib().q4_moe_block(
        _ptr(out), _ptr(x), _dtype_code(x), _ptr(logits), _ptr(W_gate), _ptr(W_up),
        _ptr(W_down), T, topk, E, H, I, _ptr(S_gate), _ptr(S_up), _ptr(S_down), Is,
        _ptr(workspace), ws_bytes, _stream(stream)))


def q4_moe_block_workspace_size(T: int, topk: int, E: int, H: int, I: int, Is: int = 0) -> int:
    return lib().q4_moe_block_workspace_size(T, topk, E, H, I, Is)


def q4_moe_static_scratch_bytes() -> int:
    return lib().q4_moe_static_scratch_bytes()


def q4_repack(dst, src, K: int, N: int, stream=None) -> None:
    _require_cuda(dst, src)
    _check("q4_repack", lib().q4_repack(_ptr(dst), _ptr(src), K, N, _stream(stream)))


def q4_unpack(dst, src, K: int, N: int, stream=None) -> None:
    _require_cuda(dst, src)
    _check("q4_unpack", lib().q4_unpack(_ptr(dst), _ptr(src), K, N, _stream(stream)))


def q4_planar_qs_offset(K: int, N: int) -> int:
    return lib().q4_planar_qs_offset(K, N)


def q4_planar_bytes(K: int, N: int) -> int:
    return lib().q4_planar_bytes(K, N)


def q4_dequant(W, B, K: int, N: int, stream=None) -> None:
    _require_cuda(W, B)
    _check("q4_dequant", lib().q4_dequant(_ptr(W), _ptr(B), K, N, _stream(stream)))


def q4_dequant_bf16(W, B, K: int, N: int, stream=None) -> None:
    _require_cuda(W, B)
    _check("q4_dequant_bf16", lib().q4_dequant_bf16(_ptr(W), _ptr(B), K, N, _stream(stream)))


def q4_selftest_wait(limit_ns: int, arrive: bool, stream=None) -> None:
    """One bounded pipeline wait run to its limit (arrive=False) or completed."""
    _check("q4_selftest_wait", lib().q4_selftest_wait(int(limit_ns), 1 if arrive else 0,
                                                      _stream(stream)))


def q4_prefill_units(M: int, N: int, K: int, sms: int):
    """The prefill form's units per CTA for this shape on `sms` SMs (host
    only): an int32 array [units, 9] of (CTA, unit, m0, n0, first K step,
    end K step, role, first helper CTA, helper count)."""
    import numpy as np
    L = lib()
    n = L.q4_prefill_units(M, N, K, sms, None, 0)
    if n < 0:
        raise Q4Error("q4_prefill_units", int(n))
    out = np.zeros((max(n, 1), 9), dtype=np.int32)
    got = L.q4_prefill_units(M, N, K, sms, out.ctypes.data, n)
    if got != n:
        raise Q4Error("q4_prefill_units", int(got))
    return out[:n]


def q4_get_device_status(stream=None) -> int:
    return lib().q4_get_device_status(_stream(stream))


def q4_last_device_flags() -> int:
    return lib().q4_last_device_flags()


def q4_version() -> int:
    return lib().q4_version()
