"""osr_softmax_rows_noalloc, the softmax entry point that allocates nothing.

Some callers cannot allocate device memory while they run (serving loops with
a frozen memory footprint, devices without stream-ordered memory pools, code
inside another allocator's callbacks).  For them the library keeps the
split-row partials in a fixed device array instead of a cudaMallocAsync
workspace.  This test calls that entry point through the C ABI, twice in a
row on each shape (the second call finds the first call's leftovers in the
shared array), and compares both outputs element by element with the fp64
oracle, within the tolerances the parity tests use.  It also covers the
in-place call (y == x), a call whose rows fill every slot of the array, and
mapped page-locked host buffers.

The file is named so that pytest collects it last."""
import ctypes

import numpy as np
import pytest
import torch

import oracle
import online_softmax_row_gb300 as osr
import workloads
from parity import check_out, to_oracle_input

pytestmark = pytest.mark.gpu

DT = {torch.float32: 0, torch.bfloat16: 1}
MAX_PARTIALS = 65536  # OSR_NOALLOC_MAX_PARTIALS in include/osr.h


def _entry():
    lib = osr.library()
    fn = lib.osr_softmax_rows_noalloc
    fn.argtypes = [ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int64, ctypes.c_int64, ctypes.c_int,
                   ctypes.c_int, ctypes.c_void_p]
    fn.restype = ctypes.c_int
    return fn


def _call(fn, x, y):
    M, N = x.shape
    return fn(x.data_ptr(), y.data_ptr(), M, N, DT[x.dtype], DT[y.dtype],
              torch.cuda.current_stream().cuda_stream)


@pytest.fixture(scope="module")
def entry():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    return _entry()


def _oracle(x_cpu):
    return oracle.softmax(to_oracle_input(x_cpu))


CASES = [
    (37, 5000, "f32", torch.float32),
    (64, 152064, "bf16", torch.float32),
    (3, 300000, "f32", torch.bfloat16),
    (1000, 1000, "bf16", torch.bfloat16),
    (5, 33, "f32", torch.float32),  # element-wise path (misaligned row length)
]


@pytest.mark.parametrize("M,N,dt,out_dtype", CASES)
def test_noalloc_matches_the_oracle_on_two_calls_in_a_row(entry, M, N, dt, out_dtype):
    x_cpu = workloads.softmax_inputs(M, N, dt, sigma=4.0, shift_rows=M // 3, seed=M + N)["x"]
    ref = _oracle(x_cpu)
    x = x_cpu.cuda()
    for _ in range(2):
        y = torch.full((M, N), float("nan"), dtype=out_dtype, device="cuda")
        assert _call(entry, x, y) == 0
        torch.cuda.synchronize()
        check_out(y, ref, f"noalloc {M}x{N} {dt}->{out_dtype}")


@pytest.mark.parametrize("M,N,dt", [(37, 5000, "f32"), (9, 152064, "bf16"), (4, 1001, "bf16")])
def test_noalloc_in_place(entry, M, N, dt):
    x_cpu = workloads.softmax_inputs(M, N, dt, sigma=4.0, shift_rows=1, seed=7 * M + N)["x"]
    ref = _oracle(x_cpu)
    for _ in range(2):
        x = x_cpu.cuda()
        assert _call(entry, x, x) == 0
        torch.cuda.synchronize()
        check_out(x, ref, f"noalloc in place {M}x{N} {dt}")


def test_noalloc_fills_every_slot_of_the_array(entry):
    # as many rows as the array has (m, d) slots, bf16 -> bf16: every slot is
    # written by pass 1 and read by pass 2
    M, N = MAX_PARTIALS, 1000
    x_cpu = workloads.softmax_inputs(M, N, "bf16", sigma=4.0, shift_rows=M // 100, seed=11)["x"]
    x = x_cpu.cuda()
    y = torch.empty(M, N, dtype=torch.bfloat16, device="cuda")
    assert _call(entry, x, y) == 0
    torch.cuda.synchronize()
    step = 8192
    for r0 in range(0, M, step):
        check_out(y[r0:r0 + step], _oracle(x_cpu[r0:r0 + step]), f"noalloc full array rows {r0}+")


def test_noalloc_rejects_more_rows_than_the_array_holds(entry):
    x = torch.zeros(MAX_PARTIALS + 1, 1, device="cuda")
    y = torch.empty_like(x)
    assert _call(entry, x, y) == 4  # OSR_ERR_UNSUPPORTED
    x = torch.randn(MAX_PARTIALS, 1, device="cuda")
    y = torch.empty_like(x)
    assert _call(entry, x, y) == 0
    torch.cuda.synchronize()
    assert torch.all(y == 1.0)


def test_noalloc_on_mapped_host_buffers(entry):
    # page-locked host buffers are accepted as osr_softmax_rows accepts them
    # (the kernels read and write them over the host link); pageable ones are
    # refused before any launch
    M, N = 6, 152064
    x_cpu = workloads.softmax_inputs(M, N, "bf16", sigma=4.0, spikes_per_row=8, seed=5)["x"]
    hx = x_cpu.clone().pin_memory()
    hy = torch.empty(M, N, dtype=torch.float32).pin_memory()
    assert _call(entry, hx, hy) == 0
    torch.cuda.synchronize()
    check_out(hy, _oracle(x_cpu), "noalloc on mapped host buffers")
    px, py = x_cpu.clone(), torch.empty(M, N, dtype=torch.float32)
    assert _call(entry, px, py) == 1  # OSR_ERR_INVALID
    assert np.isfinite(hy.numpy()).all()
