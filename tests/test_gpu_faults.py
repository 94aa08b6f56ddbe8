"""Bounded device waits report a fault instead of hanging.

The staged softmax tier waits for its bulk copies into shared memory with a
1 s bound.  A test-only entry point (osr_test_set_flags with
OSR_TEST_NO_ARRIVE, include/osr_test.h) makes that barrier receive no
arrival -- a flag nothing sets -- so the wait runs out: the kernel must
record the fault, skip its stores, leave the cluster cleanly, and the
context must keep working.  Nothing here faults, traps or hangs the GPU."""
import ctypes
import os

import pytest
import torch

import online_softmax_row_gb300 as osr
import workloads

pytestmark = pytest.mark.gpu
NO_ARRIVE = 1  # OSR_TEST_NO_ARRIVE in include/osr_test.h


def set_test_flags(flags: int) -> int:
    fn = osr.library().osr_test_set_flags
    fn.argtypes = [ctypes.c_int]
    fn.restype = ctypes.c_int
    return fn(flags)


@pytest.fixture(scope="module", autouse=True)
def gpu():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    osr.library()


@pytest.mark.parametrize("spec", ["staged:cs=2,r=0", "staged:cs=2,r=8"])
def test_wait_timeout_is_reported_and_context_survives(spec):
    # both shapes stage part of each piece in shared memory (with r=8 half of
    # it is held in registers), so every CTA waits on its copies' barriers
    assert osr.device_fault() == 0
    x = workloads.softmax_inputs(1, 32768, "f32", sigma=2.0, seed=1)["x"].cuda()
    poison = torch.full((1, 32768), 0x7FC0DEAD, dtype=torch.int32, device="cuda")
    y = poison.view(torch.float32)
    assert set_test_flags(NO_ARRIVE) == 0
    try:
        with osr.forced_kernel(spec):
            assert osr.plan_describe(osr.OP_SOFTMAX, 1, 32768, "f32").startswith("staged cs=2")
            osr.softmax_rows(x, out=y)
    finally:
        assert set_test_flags(0) == NO_ARRIVE
    assert osr.device_fault() == 1          # the bounded wait ran out and said so
    assert torch.all(poison == 0x7FC0DEAD)  # no stores after the failed wait
    assert osr.device_fault() == 0          # reading clears the word
    y2 = osr.softmax_rows(x)                # the context still works
    torch.cuda.synchronize()
    assert abs(float(y2.double().sum()) - 1.0) < 1e-4
    assert osr.device_fault() == 0
