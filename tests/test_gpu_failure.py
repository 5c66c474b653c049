"""Failure detection on the GPU without a fault: a bounded pipeline wait on a
barrier that nothing completes runs out, the device status word records the
timeout, the host reads it, and the context stays usable."""

import pytest

import oracle
import seeded_inputs as si
from gpu_util import assert_within_matmul_tol, device, to_dev, to_host64, torch

import quantized_weight_q4_gb300 as q4

pytestmark = pytest.mark.gpu


def test_wait_timeout_is_recorded_and_cleared():
    q4.q4_get_device_status()   # clear anything earlier
    q4.q4_selftest_wait(2_000_000, arrive=False)   # 2 ms limit, nothing arrives
    assert q4.q4_get_device_status() == q4.Q4_ERR_DEVICE
    assert q4.q4_last_device_flags() & q4.Q4_DEVERR_TIMEOUT
    # read-and-clear: the word is zero again
    assert q4.q4_get_device_status() == q4.Q4_OK


def test_completed_wait_records_nothing():
    q4.q4_get_device_status()
    q4.q4_selftest_wait(2_000_000, arrive=True)
    assert q4.q4_get_device_status() == q4.Q4_OK


def test_context_usable_after_timeout():
    q4.q4_selftest_wait(1_000_000, arrive=False)
    assert q4.q4_get_device_status() == q4.Q4_ERR_DEVICE
    M, K, N = 1, 512, 1024
    A = si.activations_f32(M, K, seed=12)
    B = si.q4_weights(K, N, seed=12)
    C = torch.empty((M, N), dtype=torch.float32, device=device())
    q4.q4_matmul_ex(C, to_dev(A), to_dev(B), M, N, K)
    assert q4.q4_get_device_status() == q4.Q4_OK
    C64, S = oracle.matmul(A, B, M, N, K)
    assert_within_matmul_tol(to_host64(C), C64, S, "after timeout")
