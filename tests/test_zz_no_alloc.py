"""The allocation-free routed-expert entry point.

Some callers cannot allocate device memory (a stream being captured into a
CUDA graph in global mode, loops that must not allocate after start-up, hosts
whose allocator owns all device memory).  q4_moe_experts_noalloc serves them
with scratch built into the library.  Here it is called through the C ABI
twice in a row and checked against q4_moe_experts_ex with a caller workspace
and against the oracle, within the oracle's per-element tolerance.  This file
is collected last.
"""

import ctypes

import numpy as np
import pytest

import oracle
import seeded_inputs as si
from gpu_util import device, to_dev, torch

import quantized_weight_q4_gb300 as q4

pytestmark = pytest.mark.gpu


def _inputs(T, topk, E, H, I, seed):
    Wg = np.stack([si.q4_weights(H, I, seed, 1000 + e) for e in range(E)])
    Wu = np.stack([si.q4_weights(H, I, seed, 2000 + e) for e in range(E)])
    Wd = np.stack([si.q4_weights(I, H, seed, 3000 + e) for e in range(E)])
    x = si.activations_bf16(T, H, seed)
    idx, w = si.routing(T, E, topk, seed)
    return x, Wg, Wu, Wd, idx, w


def test_noalloc_matches_workspace_entry_point():
    T, topk, E, H, I = 4, 3, 8, 512, 160
    x, Wg, Wu, Wd, idx, w = _inputs(T, topk, E, H, I, seed=21)
    dx, dg, du, dd, di, dw = (to_dev(a) for a in (x, Wg, Wu, Wd, idx, w))
    L = q4.lib()
    assert q4.q4_moe_workspace_size(T, topk, E, H, I) <= L.q4_moe_static_scratch_bytes()

    ref = torch.empty((T, H), dtype=torch.float32, device=device())
    ws = torch.zeros(q4.q4_moe_workspace_size(T, topk, E, H, I), dtype=torch.uint8,
                     device=device())
    q4.q4_moe_experts_ex(ref, dx, dg, du, dd, di, dw, T, topk, E, H, I, workspace=ws)
    torch.cuda.synchronize()
    ref_h = ref.cpu().numpy().astype(np.float64)
    want, tol, _ = oracle.moe(x, Wg, Wu, Wd, idx, w, T, topk, E, H, I)
    assert np.all(np.abs(ref_h - want) <= tol)

    stream = torch.cuda.current_stream().cuda_stream
    for _ in range(2):   # two calls in a row share the static scratch
        out = torch.full((T, H), float("nan"), dtype=torch.float32, device=device())
        rc = L.q4_moe_experts_noalloc(
            ctypes.c_void_p(out.data_ptr()), ctypes.c_void_p(dx.data_ptr()), q4.Q4_BF16,
            ctypes.c_void_p(dg.data_ptr()), ctypes.c_void_p(du.data_ptr()),
            ctypes.c_void_p(dd.data_ptr()), ctypes.c_void_p(di.data_ptr()),
            ctypes.c_void_p(dw.data_ptr()), T, topk, E, H, I, ctypes.c_void_p(stream or 0))
        assert rc == q4.Q4_OK, q4.status_str(rc)
        torch.cuda.synchronize()
        got = out.cpu().numpy().astype(np.float64)
        # the same kernels on the same inputs: within the tolerance of the
        # workspace entry point's result (in fact equal to it), and of the oracle
        assert np.all(np.abs(got - ref_h) <= tol)
        assert np.array_equal(got, ref_h)
        assert np.all(np.abs(got - want) <= tol)
    assert q4.q4_get_device_status() == q4.Q4_OK


def test_noalloc_rejects_oversized_problem():
    T, topk, E, H, I = 512, 6, 160, 5120, 1536   # needs ~80 MB of scratch
    assert q4.q4_moe_workspace_size(T, topk, E, H, I) > q4.q4_moe_static_scratch_bytes()
    z = torch.zeros(16, dtype=torch.uint8, device=device())
    rc = q4.lib().q4_moe_experts_noalloc(
        ctypes.c_void_p(z.data_ptr()), ctypes.c_void_p(z.data_ptr()), q4.Q4_BF16,
        ctypes.c_void_p(z.data_ptr()), ctypes.c_void_p(z.data_ptr()),
        ctypes.c_void_p(z.data_ptr()), ctypes.c_void_p(z.data_ptr()),
        ctypes.c_void_p(z.data_ptr()), T, topk, E, H, I, None)
    assert rc == q4.Q4_ERR_WORKSPACE
