"""GB300 (sm_103a) row-wise reduce-then-rescale: RMSNorm, fused residual-add
+ RMSNorm, and safe softmax by the online (m, d) normaliser.

Thin ctypes binding over the C ABI in ``include/osr.h`` (libosr.so, built
in-tree by ``online_softmax_row_gb300.build``).  This module only marshals
torch CUDA tensors (pointers, sizes, dtype codes, the current stream); every
step of the computation runs in the library's CUDA kernels.  There is no
fallback: if the library is not built, or an argument is rejected, a call
raises ``OsrError``.

Python name          C entry point
rmsnorm_fwd          osr_rmsnorm_fwd
layernorm_fwd        osr_layernorm_fwd
fused_add_rmsnorm    osr_fused_add_rmsnorm
softmax_rows         osr_softmax_rows
softmax_rows_stats   osr_softmax_rows_stats
log_softmax_rows     osr_log_softmax_rows
row_logsumexp        osr_row_logsumexp
row_topk             osr_row_topk
plan_describe        osr_plan_describe
bench_copy           osr_bench_copy
bench_memcpy         osr_bench_memcpy
device_fault         osr_device_fault
forced_kernel        osr_test_force_kernel (test support, osr_test.h)
"""
from __future__ import annotations

import contextlib
import ctypes
import os
import threading

import torch

from . import build as _build

__all__ = ["OsrError", "rmsnorm_fwd", "layernorm_fwd", "OP_LAYERNORM", "fused_add_rmsnorm", "softmax_rows", "softmax_rows_stats",
           "log_softmax_rows", "row_logsumexp", "row_topk", "OP_LOG_SOFTMAX", "OP_LOGSUMEXP",
           "OP_TOPK",
           "plan_describe", "bench_copy", "bench_memcpy", "device_fault", "forced_kernel", "library",
           "library_path", "OP_RMSNORM",
           "OP_FUSED",
           "OP_SOFTMAX"]

OP_RMSNORM, OP_FUSED, OP_SOFTMAX, OP_LOG_SOFTMAX, OP_LOGSUMEXP, OP_LAYERNORM, OP_TOPK = 0, 1, 2, 3, 4, 5, 6
_DT = {torch.float32: 0, torch.bfloat16: 1}
_DT_NAME = {"f32": 0, "bf16": 1}
_STATUS = {0: "OSR_OK", 1: "OSR_ERR_INVALID", 2: "OSR_ERR_ALIGN", 3: "OSR_ERR_ALIAS",
           4: "OSR_ERR_UNSUPPORTED", 5: "OSR_ERR_CUDA", 6: "OSR_ERR_DEVICE_TIMEOUT"}

_lock = threading.Lock()
_lib = None


class OsrError(RuntimeError):
    def __init__(self, status: int, where: str, detail: str = ""):
        self.status = status
        self.name = _STATUS.get(status, str(status))
        super().__init__(f"{where}: {self.name}{': ' + detail if detail else ''}")


def library_path() -> str:
    return _build.LIB


def library():
    """The loaded libosr.so (ctypes.CDLL).  Raises OsrError if it is not built."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        path = _build.LIB
        if not os.path.exists(path):
            raise OsrError(1, "libosr.so", f"not built at {path}; run "
                           "`python -m online_softmax_row_gb300.build`")
        lib = ctypes.CDLL(path)
        P, I64, I, F = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int, ctypes.c_float
        lib.osr_rmsnorm_fwd.argtypes = [P, P, F, P, I64, I64, I, P]
        lib.osr_fused_add_rmsnorm.argtypes = [P, P, P, F, P, I64, I64, I, P]
        lib.osr_softmax_rows.argtypes = [P, P, I64, I64, I, I, P]
        lib.osr_softmax_rows_stats.argtypes = [P, P, P, P, I64, I64, I, I, P]
        lib.osr_status_string.argtypes = [I]
        lib.osr_status_string.restype = ctypes.c_char_p
        lib.osr_last_cuda_error.restype = I
        lib.osr_plan_describe.argtypes = [I, I64, I64, I, I, I, I, ctypes.c_char_p, ctypes.c_size_t]
        lib.osr_version.restype = I
        lib.osr_bench_copy.argtypes = [P, P, ctypes.c_size_t, P]
        lib.osr_bench_memcpy.argtypes = [P, P, ctypes.c_size_t, P]
        lib.osr_device_fault.argtypes = [P, ctypes.POINTER(I)]
        lib.osr_log_softmax_rows.argtypes = [P, P, I64, I64, I, I, P]
        lib.osr_layernorm_fwd.argtypes = [P, P, P, F, P, I64, I64, I, P]
        lib.osr_row_logsumexp.argtypes = [P, P, P, I64, I64, I, P]
        lib.osr_row_topk.argtypes = [P, P, P, P, P, I64, I64, I64, I, P]
        lib.osr_test_force_kernel.argtypes = [ctypes.c_char_p]
        for fn in ("osr_rmsnorm_fwd", "osr_fused_add_rmsnorm", "osr_softmax_rows",
                   "osr_softmax_rows_stats", "osr_plan_describe", "osr_bench_copy", "osr_bench_memcpy",
                   "osr_device_fault", "osr_log_softmax_rows", "osr_row_logsumexp", "osr_row_topk",
                   "osr_layernorm_fwd", "osr_test_force_kernel"):
            getattr(lib, fn).restype = I
        _lib = lib
        return lib


def _check(status: int, where: str):
    if status != 0:
        lib = library()
        detail = lib.osr_status_string(status).decode()
        if status == 5:
            detail += f" (cudaError {lib.osr_last_cuda_error()})"
        raise OsrError(status, where, detail)


_raw_stream_fn = getattr(torch._C, "_cuda_getCurrentRawStream", None)


def _raw_stream(index: int) -> int:
    """cudaStream_t of torch's current stream on device `index`."""
    if _raw_stream_fn is not None:
        return _raw_stream_fn(index)
    return torch.cuda.current_stream(index).cuda_stream


def _run(t: torch.Tensor, fn, *args):
    """Call a C entry point with the tensor's device current and its current
    stream appended as the last argument."""
    index = t.device.index
    if index is None or index == torch.cuda.current_device():
        return fn(*args, _raw_stream(torch.cuda.current_device() if index is None else index))
    with torch.cuda.device(index):
        return fn(*args, _raw_stream(index))


def _rows(t: torch.Tensor, name: str):
    if not t.is_cuda:
        raise OsrError(1, name, "expected a CUDA tensor")
    if t.dtype not in _DT:
        raise OsrError(1, name, f"dtype {t.dtype} (float32 or bfloat16 expected)")
    if not t.is_contiguous():
        raise OsrError(1, name, "expected a contiguous (row-major) tensor")
    if t.dim() == 0:
        raise OsrError(1, name, "expected at least one dimension")
    n = t.shape[-1]
    m = t.numel() // n if n else 0
    return m, n


def rmsnorm_fwd(x: torch.Tensor, gamma: torch.Tensor, eps: float = 1e-6,
                out: torch.Tensor | None = None) -> torch.Tensor:
    """y = x * rsqrt(mean(x^2, -1) + eps) * gamma over the last dimension."""
    M, H = _rows(x, "x")
    if gamma.shape != (H,) or gamma.dtype != x.dtype:
        raise OsrError(1, "gamma", f"expected shape ({H},) and dtype {x.dtype}")
    _rows(gamma, "gamma")
    if out is None:
        out = torch.empty_like(x)
    elif out.shape != x.shape or out.dtype != x.dtype:
        raise OsrError(1, "out", "shape/dtype must match x")
    _rows(out, "out")
    lib = _lib or library()
    _check(_run(x, lib.osr_rmsnorm_fwd, x.data_ptr(), gamma.data_ptr(), float(eps), out.data_ptr(),
                M, H, _DT[x.dtype]), "osr_rmsnorm_fwd")
    return out


def layernorm_fwd(x: torch.Tensor, gamma: torch.Tensor, beta: torch.Tensor, eps: float = 1e-5,
                  out: torch.Tensor | None = None) -> torch.Tensor:
    """y = (x - mean) / sqrt(var + eps) * gamma + beta over the last dimension."""
    M, H = _rows(x, "x")
    for name, t in (("gamma", gamma), ("beta", beta)):
        if t.shape != (H,) or t.dtype != x.dtype:
            raise OsrError(1, name, f"expected shape ({H},) and dtype {x.dtype}")
        _rows(t, name)
    if out is None:
        out = torch.empty_like(x)
    elif out.shape != x.shape or out.dtype != x.dtype:
        raise OsrError(1, "out", "shape/dtype must match x")
    _rows(out, "out")
    lib = _lib or library()
    _check(_run(x, lib.osr_layernorm_fwd, x.data_ptr(), gamma.data_ptr(), beta.data_ptr(),
                float(eps), out.data_ptr(), M, H, _DT[x.dtype]), "osr_layernorm_fwd")
    return out


def fused_add_rmsnorm(x: torch.Tensor, residual: torch.Tensor, gamma: torch.Tensor,
                      eps: float = 1e-6, out: torch.Tensor | None = None) -> torch.Tensor:
    """residual <- x + residual (in place); returns RMSNorm(residual) * gamma."""
    M, H = _rows(x, "x")
    if residual.shape != x.shape or residual.dtype != x.dtype:
        raise OsrError(1, "residual", "shape/dtype must match x")
    _rows(residual, "residual")
    if gamma.shape != (H,) or gamma.dtype != x.dtype:
        raise OsrError(1, "gamma", f"expected shape ({H},) and dtype {x.dtype}")
    _rows(gamma, "gamma")
    if out is None:
        out = torch.empty_like(x)
    elif out.shape != x.shape or out.dtype != x.dtype:
        raise OsrError(1, "out", "shape/dtype must match x")
    _rows(out, "out")
    lib = _lib or library()
    _check(_run(x, lib.osr_fused_add_rmsnorm, x.data_ptr(), residual.data_ptr(), gamma.data_ptr(),
                float(eps), out.data_ptr(), M, H, _DT[x.dtype]), "osr_fused_add_rmsnorm")
    return out


def _softmax_out(x, out, out_dtype):
    if out is None:
        out = torch.empty(x.shape, dtype=out_dtype or x.dtype, device=x.device)
    elif out.shape != x.shape or (out_dtype is not None and out.dtype != out_dtype):
        raise OsrError(1, "out", "shape must match x (and dtype out_dtype)")
    _rows(out, "out")
    return out


def softmax_rows(x: torch.Tensor, out: torch.Tensor | None = None,
                 out_dtype: torch.dtype | None = None) -> torch.Tensor:
    """Softmax over the last dimension (float32 or bfloat16 in and out)."""
    M, N = _rows(x, "x")
    out = _softmax_out(x, out, out_dtype)
    lib = _lib or library()
    _check(_run(x, lib.osr_softmax_rows, x.data_ptr(), out.data_ptr(), M, N, _DT[x.dtype],
                _DT[out.dtype]), "osr_softmax_rows")
    return out


def softmax_rows_stats(x: torch.Tensor, out: torch.Tensor | None = None,
                       out_dtype: torch.dtype | None = None):
    """Softmax plus each row's (max, sum of exp(x - max)) as float32 tensors."""
    M, N = _rows(x, "x")
    out = _softmax_out(x, out, out_dtype)
    lead = x.shape[:-1]
    row_max = torch.empty(lead, dtype=torch.float32, device=x.device)
    row_sum = torch.empty(lead, dtype=torch.float32, device=x.device)
    lib = _lib or library()
    _check(_run(x, lib.osr_softmax_rows_stats, x.data_ptr(), out.data_ptr(), row_max.data_ptr(),
                row_sum.data_ptr(), M, N, _DT[x.dtype], _DT[out.dtype]), "osr_softmax_rows_stats")
    return out, row_max, row_sum


def log_softmax_rows(x: torch.Tensor, out: torch.Tensor | None = None,
                     out_dtype: torch.dtype | None = None) -> torch.Tensor:
    """Log-softmax over the last dimension: (x - max) - log(sum exp(x - max))."""
    M, N = _rows(x, "x")
    out = _softmax_out(x, out, out_dtype)
    lib = _lib or library()
    _check(_run(x, lib.osr_log_softmax_rows, x.data_ptr(), out.data_ptr(), M, N, _DT[x.dtype],
                _DT[out.dtype]), "osr_log_softmax_rows")
    return out


def row_logsumexp(x: torch.Tensor, want_lse: bool = True, want_argmax: bool = True):
    """Per row: log(sum exp(x)) (float32) and the first index of the maximum
    (int64), reading x once and writing nothing else."""
    M, N = _rows(x, "x")
    lead = x.shape[:-1]
    lse = torch.empty(lead, dtype=torch.float32, device=x.device) if want_lse else None
    am = torch.empty(lead, dtype=torch.int64, device=x.device) if want_argmax else None
    lib = _lib or library()
    _check(_run(x, lib.osr_row_logsumexp, x.data_ptr(), lse.data_ptr() if lse is not None else None,
                am.data_ptr() if am is not None else None, M, N, _DT[x.dtype]), "osr_row_logsumexp")
    return lse, am


def row_topk(x: torch.Tensor, k: int, want_probs: bool = True, want_lse: bool = True):
    """Per row: the k largest values (float32, largest first, equal values by
    column), their column indices (int64), the softmax of those k values
    (float32) and the row's log-sum-exp (float32), reading x once.  Returns
    (values, indices, probs or None, lse or None); leading dimensions of x
    are kept."""
    M, N = _rows(x, "x")
    lead = x.shape[:-1]
    values = torch.empty(*lead, k, dtype=torch.float32, device=x.device)
    indices = torch.empty(*lead, k, dtype=torch.int64, device=x.device)
    probs = torch.empty(*lead, k, dtype=torch.float32, device=x.device) if want_probs else None
    lse = torch.empty(lead, dtype=torch.float32, device=x.device) if want_lse else None
    lib = _lib or library()
    _check(_run(x, lib.osr_row_topk, x.data_ptr(), values.data_ptr(), indices.data_ptr(),
                probs.data_ptr() if probs is not None else None,
                lse.data_ptr() if lse is not None else None, M, N, int(k), _DT[x.dtype]),
           "osr_row_topk")
    return values, indices, probs, lse


def plan_describe(op: int, M: int, N: int, in_dtype: str = "f32", out_dtype: str | None = None,
                  vec_ok: bool = True, sm_count: int = 152) -> str:
    """Kernel the dispatcher picks for a shape (host-only, no GPU needed)."""
    buf = ctypes.create_string_buffer(128)
    _check(library().osr_plan_describe(op, M, N, _DT_NAME[in_dtype], _DT_NAME[out_dtype or in_dtype],
                                       int(vec_ok), sm_count, buf, 128), "osr_plan_describe")
    return buf.value.decode()


def bench_copy(src: torch.Tensor, dst: torch.Tensor) -> None:
    """dst <- src bytes with the library's 128-bit copy kernel (HBM peak probe)."""
    nbytes = src.numel() * src.element_size()
    if dst.numel() * dst.element_size() != nbytes:
        raise OsrError(1, "bench_copy", "sizes differ")
    _check(_run(src, library().osr_bench_copy, src.data_ptr(), dst.data_ptr(), nbytes),
           "osr_bench_copy")


def bench_memcpy(src: torch.Tensor, dst: torch.Tensor) -> None:
    """dst <- src bytes by the runtime's device-to-device memcpy (HBM peak probe)."""
    nbytes = src.numel() * src.element_size()
    if dst.numel() * dst.element_size() != nbytes:
        raise OsrError(1, "bench_memcpy", "sizes differ")
    _check(_run(src, library().osr_bench_memcpy, src.data_ptr(), dst.data_ptr(), nbytes),
           "osr_bench_memcpy")


def device_fault(device=None) -> int:
    """Synchronise the current stream and return (and clear) the device's
    fault word: 0 if no kernel's bounded wait has run out since the last call."""
    dev = torch.device("cuda", torch.cuda.current_device()) if device is None else torch.device(device)
    v = ctypes.c_int(0)
    with torch.cuda.device(dev):
        st = library().osr_device_fault(torch.cuda.current_stream(dev).cuda_stream, ctypes.byref(v))
    if st not in (0, 6):
        _check(st, "osr_device_fault")
    return v.value


@contextlib.contextmanager
def forced_kernel(spec: str | None):
    """Test support: every call inside the block (and plan_describe) uses the
    forced plan `spec` (e.g. "rows:g=512", "staged:cs=3,r=8", "lse:g=32",
    "topk:cs=8"; see include/osr_test.h); None or "" forces nothing.  The
    previous state, none, is restored on exit."""
    lib = library()
    _check(lib.osr_test_force_kernel(spec.encode() if spec else None), "osr_test_force_kernel")
    try:
        yield
    finally:
        lib.osr_test_force_kernel(None)
