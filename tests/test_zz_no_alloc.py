"""osr_softmax_rows_noalloc, the softmax entry point that allocates nothing.

Some callers cannot allocate device memory while they run (serving loops with
a frozen memory footprint, devices without stream-ordered memory pools, code
inside another allocator's callbacks).  For them the library keeps the
split-row partials in a fixed device array instead of a cudaMallocAsync
workspace.  This test calls that entry point through the C ABI, twice in a
row on each shape (the second call finds the first call's leftovers in the
shared array), and compares both outputs with what osr_softmax_rows returns
for the same input, within the tolerances the parity tests use.

The file is named so that pytest collects it last."""
import ctypes

import pytest
import torch

import online_softmax_row_gb300 as osr
import workloads
from parity import check_bf16, check_f32

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


CASES = [
    (37, 5000, "f32", torch.float32),
    (64, 152064, "bf16", torch.float32),
    (3, 300000, "f32", torch.bfloat16),
    (1000, 1000, "bf16", torch.bfloat16),
    (5, 33, "f32", torch.float32),  # element-wise path (misaligned row length)
]


@pytest.mark.parametrize("M,N,dt,out_dtype", CASES)
def test_noalloc_matches_softmax_rows_on_two_calls_in_a_row(entry, M, N, dt, out_dtype):
    x = workloads.softmax_inputs(M, N, dt, sigma=4.0, shift_rows=M // 3, seed=M + N)["x"].cuda()
    ref = osr.softmax_rows(x, out_dtype=out_dtype).double().cpu().numpy()
    for _ in range(2):
        y = torch.full((M, N), float("nan"), dtype=out_dtype, device="cuda")
        assert _call(entry, x, y) == 0
        torch.cuda.synchronize()
        if out_dtype == torch.float32:
            check_f32(y, ref, "noalloc vs softmax_rows")
        else:
            check_bf16(y, ref, "noalloc vs softmax_rows")


def test_noalloc_rejects_more_rows_than_the_array_holds(entry):
    x = torch.zeros(MAX_PARTIALS + 1, 1, device="cuda")
    y = torch.empty_like(x)
    assert _call(entry, x, y) == 4  # OSR_ERR_UNSUPPORTED
    x = torch.randn(MAX_PARTIALS, 1, device="cuda")
    y = torch.empty_like(x)
    assert _call(entry, x, y) == 0
    torch.cuda.synchronize()
    assert torch.all(y == 1.0)
