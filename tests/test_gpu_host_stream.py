"""Host-streamed weights: a sequence of matmuls whose Q4_0 weights stay in
pinned host memory and are copied into a ring of device slots while earlier
matmuls run.  Each result must equal, bit for bit, the same matmul run from a
device copy of the weights (same kernel, same bytes, deterministic), and one
of them is checked against the oracle as well.
"""

import numpy as np
import pytest

import oracle
import seeded_inputs as si
from gpu_util import assert_within_matmul_tol, device, to_dev, to_host64, torch

import quantized_weight_q4_gb300 as q4

pytestmark = pytest.mark.gpu

SHAPES = [(1, 4096, 4096), (2, 333, 300), (1, 1000, 1056), (3, 64, 96), (1, 2048, 11008),
          (4, 515, 800), (1, 4096, 4096)]


def make_ops(shapes, seed=0, bf16_every=3):
    ops, ref = [], []
    for i, (M, K, N) in enumerate(shapes):
        A = (si.activations_bf16(M, K, seed=seed + i) if i % bf16_every == 1
             else si.activations_f32(M, K, seed=seed + i))
        B = si.q4_weights(K, N, seed=seed + i, stream=7)
        dA = to_dev(A)
        C = torch.empty((M, N), dtype=torch.float32, device=device())
        Bh = torch.from_numpy(B).pin_memory()
        ops.append((C, dA, Bh, M, N, K))
        Cref = torch.empty_like(C)
        q4.q4_matmul_ex(Cref, dA, to_dev(B), M, N, K)
        ref.append(Cref)
    torch.cuda.synchronize()
    return ops, ref


def staging_for(ops, slots):
    nbytes = q4.q4_host_stream_slot_bytes(ops) * slots
    return torch.empty(nbytes, dtype=torch.uint8, device=device())


@pytest.mark.parametrize("slots", [1, 2, 3, 16])
def test_results_equal_device_resident_runs(slots):
    ops, ref = make_ops(SHAPES)
    st, cp = torch.cuda.Stream(), torch.cuda.Stream()
    with torch.cuda.stream(st):
        q4.q4_matmul_host_stream(ops, staging_for(ops, slots), slots, stream=st, copy_stream=cp)
    st.synchronize()
    for (C, *_), R in zip(ops, ref):
        assert torch.equal(C, R)
    assert q4.q4_get_device_status() == q4.Q4_OK


def test_one_result_against_the_oracle():
    M, K, N = 1, 4096, 4096
    ops, _ = make_ops([(M, K, N)], seed=5)
    st, cp = torch.cuda.Stream(), torch.cuda.Stream()
    q4.q4_matmul_host_stream(ops, staging_for(ops, 2), 2, stream=st, copy_stream=cp)
    st.synchronize()
    A = si.activations_f32(M, K, seed=5)
    B = si.q4_weights(K, N, seed=5, stream=7)
    C64, S = oracle.matmul(A, B, M, N, K)
    assert_within_matmul_tol(to_host64(ops[0][0]), C64, S, "host-streamed 4096x4096")


def test_stream_order_before_and_after():
    """Work enqueued on the stream before the call (writing A) is seen by the
    first matmul; work after it (a copy of C) sees the last result."""
    ops, ref = make_ops(SHAPES[:3], seed=11)
    st, cp = torch.cuda.Stream(), torch.cuda.Stream()
    A0 = ops[0][1]
    saved = A0.clone()
    A0.zero_()
    torch.cuda.synchronize()
    out = torch.empty_like(ops[-1][0])
    with torch.cuda.stream(st):
        A0.copy_(saved)   # on `st`, before the sequence
        q4.q4_matmul_host_stream(ops, staging_for(ops, 2), 2, stream=st, copy_stream=cp)
        out.copy_(ops[-1][0])   # on `st`, after it
    st.synchronize()
    assert torch.equal(ops[0][0], ref[0])
    assert torch.equal(out, ref[-1])


def test_graph_capture_replays_the_sequence():
    ops, ref = make_ops(SHAPES, seed=3)
    staging = staging_for(ops, 3)
    st, cp = torch.cuda.Stream(), torch.cuda.Stream()
    q4.q4_matmul_host_stream(ops, staging, 3, stream=st, copy_stream=cp)   # warm the shape cache
    st.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=st):
        q4.q4_matmul_host_stream(ops, staging, 3, stream=st, copy_stream=cp)
    for C, *_ in ops:
        C.zero_()
    torch.cuda.synchronize()
    g.replay()
    torch.cuda.synchronize()
    for (C, *_), R in zip(ops, ref):
        assert torch.equal(C, R)


def test_rejections():
    ops, _ = make_ops(SHAPES[:2], seed=2)
    st, cp = torch.cuda.Stream(), torch.cuda.Stream()
    small = torch.empty(q4.q4_host_stream_slot_bytes(ops) * 2 - 256, dtype=torch.uint8,
                        device=device())
    with pytest.raises(q4.Q4Error) as e:
        q4.q4_matmul_host_stream(ops, small, 2, stream=st, copy_stream=cp)
    assert e.value.status == q4.Q4_ERR_WORKSPACE
    with pytest.raises(q4.Q4Error) as e:
        q4.q4_matmul_host_stream(ops, staging_for(ops, 2), 2, stream=st, copy_stream=st)
    assert e.value.status == q4.Q4_ERR_ARG
    # B in pageable host memory is refused
    C, A, Bh, M, N, K = ops[1]
    pageable = torch.from_numpy(np.ascontiguousarray(Bh.numpy().copy()))
    with pytest.raises(q4.Q4Error) as e:
        q4.q4_matmul_host_stream([ops[0], (C, A, pageable, M, N, K)], staging_for(ops, 2), 2,
                                 stream=st, copy_stream=cp)
    assert e.value.status == q4.Q4_ERR_ARG
    st.synchronize()
