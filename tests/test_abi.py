"""The C ABI library loads, exports every function include/q4.h declares, and
rejects bad arguments on the host (no GPU needed: none of these calls reaches
a CUDA API)."""

import ctypes
import os
import re

import pytest

import quantized_weight_q4_gb300 as q4
from quantized_weight_q4_gb300 import _build

HEADER = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "include", "q4.h")


@pytest.fixture(scope="module")
def L():
    _build.build()
    return q4.lib()


def declared_functions():
    with open(HEADER) as f:
        text = f.read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"Q4_API\s+[\w\s\*]+?\b(q4_\w+)\s*\(", text)))


def test_header_declares_entry_points():
    names = declared_functions()
    for must in ("q4_matmul", "q4_moe_experts", "q4_repack", "q4_unpack", "q4_dequant"):
        assert must in names


def test_every_declared_symbol_is_exported(L):
    names = declared_functions()
    assert names
    for n in names:
        assert hasattr(L, n), n
        assert n in q4.SIGNATURES, f"binding lacks {n}"


def test_binding_has_no_extra_symbols():
    assert set(q4.SIGNATURES) == set(declared_functions())


def test_status_strings(L):
    for code in (0, -1, -2, -3, -4, -5, -6, -7):
        assert q4.status_str(code)
    assert q4.status_str(-99) == "unknown status"
    assert L.q4_version() >= 100


def test_planar_sizes(L):
    # K = 3, N = 40: nb = 2, 6 blocks: scales 12 bytes -> qs from 16, 96 qs bytes
    assert L.q4_planar_qs_offset(3, 40) == 16
    assert L.q4_planar_bytes(3, 40) == 16 + 6 * 16
    assert L.q4_planar_bytes(0, 40) == 0


def test_argument_errors_on_host(L):
    vp = ctypes.c_void_p
    good = vp(0x10000)
    # null pointers and non-positive sizes
    assert L.q4_matmul(None, good, good, 1, 32, 32) == q4.Q4_ERR_ARG
    assert L.q4_matmul(good, good, good, 0, 32, 32) == q4.Q4_ERR_ARG
    assert L.q4_matmul(good, good, good, 1, -5, 32) == q4.Q4_ERR_ARG
    # bad dtype and layout codes
    assert L.q4_matmul_ex(good, 7, good, 0, good, 0, 1, 32, 32, None, 0, None) == q4.Q4_ERR_DTYPE
    assert L.q4_matmul_ex(good, 0, good, 0, good, 9, 1, 32, 32, None, 0, None) == q4.Q4_ERR_ARG
    # sizes beyond 2^30 are shape errors for every layout (checked before any
    # CUDA call)
    for layout in (q4.Q4_LAYOUT_BLOCKS, q4.Q4_LAYOUT_Q8_0, q4.Q4_LAYOUT_PLANAR):
        assert L.q4_matmul_ex(good, 0, good, 0, good, layout, (1 << 30) + 1, 32, 32, None, 0,
                              None) == q4.Q4_ERR_SHAPE
    # misaligned pointers
    bad = vp(0x10004)
    assert L.q4_matmul(bad, good, good, 1, 32, 32) == q4.Q4_ERR_ALIGN
    assert L.q4_matmul(good, good, bad, 1, 32, 32) == q4.Q4_ERR_ALIGN
    # experts
    args = [good] * 7
    assert L.q4_moe_experts(None, *args[1:], 1, 160, 5120, 1536) == q4.Q4_ERR_ARG
    assert L.q4_moe_experts(*args, 0, 160, 5120, 1536) == q4.Q4_ERR_ARG
    assert L.q4_moe_experts_ex(*args[:2], 0, *args[2:], 1, 17, 160, 5120, 1536, None, 0,
                               None) == q4.Q4_ERR_SHAPE
    assert L.q4_moe_experts_ex(*args[:2], 5, *args[2:], 1, 6, 160, 5120, 1536, None, 0,
                               None) == q4.Q4_ERR_DTYPE
    assert L.q4_repack(bad, good, 4, 64, None) == q4.Q4_ERR_ALIGN
    assert L.q4_dequant(good, good, 0, 64, None) == q4.Q4_ERR_ARG
    # the failure-detection self-test checks its limit and mode before any CUDA call
    for limit, arrive in [(0, 0), (-5, 0), (2_000_000_000, 0), (1000, 2)]:
        assert L.q4_selftest_wait(limit, arrive, None) == q4.Q4_ERR_ARG


def test_host_stream_checks_on_host(L):
    """The host-streamed sequence checks every op before any CUDA call."""
    vp = ctypes.c_void_p
    good, bad = 0x10000, 0x10004
    ops = (q4.SeqOp * 2)(q4.SeqOp(good, good, good, 1, 64, 32, 0, 0),
                         q4.SeqOp(good, good, good, 2, 40, 96, 1, 0))
    # slot: the larger B, 96 x 2 blocks x 18 = 3456 -> 3584 (256-byte rounding)
    assert L.q4_host_stream_slot_bytes(ops, 2) == 3584
    assert L.q4_host_stream_slot_bytes(ops, 0) == 0
    s1, s2 = vp(0x1000), vp(0x2000)
    assert L.q4_matmul_host_stream(None, 2, vp(good), 1 << 20, 2, s1, s2) == q4.Q4_ERR_ARG
    assert L.q4_matmul_host_stream(ops, 2, vp(good), 1 << 20, 0, s1, s2) == q4.Q4_ERR_ARG
    assert L.q4_matmul_host_stream(ops, 2, vp(good), 1 << 20, 2, s1, s1) == q4.Q4_ERR_ARG
    assert L.q4_matmul_host_stream(ops, 2, vp(good + 16), 1 << 20, 2, s1, s2) == q4.Q4_ERR_ALIGN
    assert L.q4_matmul_host_stream(ops, 2, vp(good), 3584, 2, s1, s2) == q4.Q4_ERR_WORKSPACE
    ops[1].K = 0
    assert L.q4_matmul_host_stream(ops, 2, vp(good), 1 << 20, 2, s1, s2) == q4.Q4_ERR_ARG
    ops[1].K, ops[1].a_dtype = 96, 3
    assert L.q4_matmul_host_stream(ops, 2, vp(good), 1 << 20, 2, s1, s2) == q4.Q4_ERR_DTYPE
    ops[1].a_dtype, ops[1].C = 1, bad
    assert L.q4_matmul_host_stream(ops, 2, vp(good), 1 << 20, 2, s1, s2) == q4.Q4_ERR_ALIGN


def test_gemv_seq_checks_on_host(L):
    """The decode sequence checks every op, and the plan buffer, before any
    CUDA call; its buffer holds 2 KB of partial sums per unit (512 columns
    of 64 to 4096 rows), which shows how many units the plan has."""
    vp = ctypes.c_void_p
    good = 0x10000

    def op(N, K, deps=(), a=0, c=0, C=good, rows=512):
        d = (ctypes.c_int * 4)(*(list(deps) + [0] * (4 - len(deps))))
        return q4.GemvOp(C, good, good, N, K, a, c, len(deps), d, rows)

    ops = (q4.GemvOp * 3)(op(4096, 4096), op(11008, 4096, [0]), op(4096, 11008, [0, 1]))
    units = 8 * 8 + 22 * 8 + 8 * 22
    nbytes = L.q4_gemv_seq_bytes(ops, 3)
    assert units * 2048 < nbytes < units * 2048 + 65536
    # the library's choice: 512 rows for ops 0 and 1, which op 2 waits for,
    # and for op 2, the whole sequence being under one half-round of 1024-row
    # units (0.5 x 304 CTAs x 1024 rows x 288 bytes = 44.8 MB)
    auto = (q4.GemvOp * 3)(op(4096, 4096, rows=0), op(11008, 4096, [0], rows=0),
                           op(4096, 11008, [0, 1], rows=0))
    units_auto = 8 * 8 + 22 * 8 + 8 * 22
    assert units_auto * 2048 < L.q4_gemv_seq_bytes(auto, 3) < units_auto * 2048 + 65536
    # ten independent (K = 11008, N = 4096) ops of 25,362,432 weight bytes:
    # counted from the end, units of 512 rows while under 44.8 MB remain
    # (1 op), 1024 under 89.7 MB (2), 2048 under 179.3 MB (4), then 4096 (3)
    graded = (q4.GemvOp * 10)(*[op(4096, 11008, rows=0) for _ in range(10)])
    units_graded = 8 * (3 * 3 + 4 * 6 + 2 * 11 + 1 * 22)
    assert units_graded * 2048 < L.q4_gemv_seq_bytes(graded, 10) < units_graded * 2048 + 65536
    short = (q4.GemvOp * 3)(op(4096, 4096, rows=128), op(11008, 4096, [0], rows=128),
                            op(4096, 11008, [0, 1], rows=128))
    units_short = 8 * 32 + 22 * 32 + 8 * 86
    assert units_short * 2048 < L.q4_gemv_seq_bytes(short, 3) < units_short * 2048 + 65536
    # a unit may end on half of a 128-row stage: 64 and 192 rows stay valid
    for r in (64, 192):
        half = (q4.GemvOp * 1)(op(4096, 4096, rows=r))
        units_half = 8 * -(-4096 // r)
        assert units_half * 2048 < L.q4_gemv_seq_bytes(half, 1) < units_half * 2048 + 65536
    plan = vp()
    create = lambda o, n, buf, size: L.q4_gemv_seq_create(o, n, vp(buf), size, ctypes.byref(plan))
    assert create(ops, 3, good + 16, nbytes) == q4.Q4_ERR_ALIGN
    assert create(ops, 3, good, nbytes - 1) == q4.Q4_ERR_WORKSPACE
    assert create(ops, 0, good, nbytes) == q4.Q4_ERR_ARG
    assert L.q4_gemv_seq_bytes(ops, 0) == 0
    cases = [((op(4096, 4096), op(4096, 4096, [1])), q4.Q4_ERR_ARG),     # not an earlier op
             ((op(4096, 4096, [-1]),), q4.Q4_ERR_ARG),
             ((op(100, 64),), q4.Q4_ERR_SHAPE),                          # 4 blocks per row
             ((op(256, 64, a=3),), q4.Q4_ERR_DTYPE),
             ((op(256, 0),), q4.Q4_ERR_ARG),
             ((op(256, 64, C=good + 4),), q4.Q4_ERR_ALIGN),
             ((op(256, 64, rows=100),), q4.Q4_ERR_ARG),                  # not a multiple of 64
             ((op(256, 64, rows=4160),), q4.Q4_ERR_ARG)]     # over 4096
    for bad, code in cases:
        arr = (q4.GemvOp * len(bad))(*bad)
        assert L.q4_gemv_seq_bytes(arr, len(bad)) == 0
        assert create(arr, len(bad), good, 1 << 30) == code
    assert plan.value is None
