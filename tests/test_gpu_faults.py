"""Bounded device waits report a fault instead of hanging.

The staged softmax tier waits for its bulk copies into shared memory with a
1 s bound.  A test hook (OSR_TEST_HOOK=no_arrive) makes that barrier receive
no arrival -- a flag nothing sets -- so the wait runs out: the kernel must
record the fault, skip its stores, leave the cluster cleanly, and the
context must keep working.  Nothing here faults, traps or hangs the GPU."""
import os

import pytest
import torch

import online_softmax_row_gb300 as osr
import workloads

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def gpu():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    osr.library()


def test_wait_timeout_is_reported_and_context_survives():
    assert osr.device_fault() == 0
    x = workloads.softmax_inputs(1, 32768, "f32", sigma=2.0, seed=1)["x"].cuda()
    assert osr.plan_describe(osr.OP_SOFTMAX, 1, 32768, "f32").startswith("staged")
    poison = torch.full((1, 32768), 0x7FC0DEAD, dtype=torch.int32, device="cuda")
    y = poison.view(torch.float32)
    os.environ["OSR_TEST_HOOK"] = "no_arrive"
    try:
        osr.softmax_rows(x, out=y)
    finally:
        del os.environ["OSR_TEST_HOOK"]
    assert osr.device_fault() == 1          # the bounded wait ran out and said so
    assert torch.all(poison == 0x7FC0DEAD)  # no stores after the failed wait
    assert osr.device_fault() == 0          # reading clears the word
    y2 = osr.softmax_rows(x)                # the context still works
    torch.cuda.synchronize()
    assert abs(float(y2.double().sum()) - 1.0) < 1e-4
    assert osr.device_fault() == 0
