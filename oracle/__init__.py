"""fp64 CPU oracle for RMSNorm, fused residual-add + RMSNorm and safe softmax.

TEST INFRASTRUCTURE.  Only ``tests/``, ``__graft_entry__.smoke()`` and the
``cpu_baseline`` / ``--impl reference`` legs of ``bench.py`` may import this
package.  The product library (``online_softmax_row_gb300``) never imports it,
and this package imports nothing from the product.

The arithmetic lives in ``oracle.c`` (plain C, binary64); this module only
builds that file with gcc and marshals numpy arrays through ctypes.  Inputs
are numpy arrays: ``float32`` for binary32 data, ``uint16`` holding the raw
bit patterns for bfloat16 data.  Outputs are ``float64`` arrays.

Parity status: pinned (worked examples printed on the pages, closed forms,
invariants and library cross-checks in ``tests/test_oracle.py``).
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

HERE = os.path.dirname(os.path.abspath(__file__))
SRC = os.path.join(HERE, "oracle.c")
BUILD_DIR = os.path.join(HERE, "_build")
LIB = os.path.join(BUILD_DIR, "liboracle.so")

F32, BF16 = 0, 1
_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile oracle.c with gcc (-O2, no fast-math) into oracle/_build."""
    os.makedirs(BUILD_DIR, exist_ok=True)
    if force or not os.path.exists(LIB) or os.path.getmtime(LIB) < os.path.getmtime(SRC):
        tmp = LIB + f".tmp{os.getpid()}"
        cmd = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-fopenmp", SRC, "-o", tmp, "-lm"]
        subprocess.run(cmd, check=True)
        os.replace(tmp, LIB)
    return LIB


def _configure(lib):
        P = ctypes.c_void_p
        I64 = ctypes.c_int64
        D = ctypes.c_double
        I = ctypes.c_int
        lib.orc_set_threads.argtypes = [I]
        lib.orc_get_threads.restype = I
        lib.orc_round_bf16.argtypes = [D]
        lib.orc_round_bf16.restype = ctypes.c_uint16
        lib.orc_round_array.argtypes = [P, I64, I, P]
        lib.orc_rmsnorm.argtypes = [P, P, I, D, I64, I64, P, P]
        lib.orc_fused_add_rmsnorm.argtypes = [P, P, P, I, D, I64, I64, P, P, P]
        lib.orc_softmax.argtypes = [P, I, I64, I64, P, P, P]
        lib.orc_softmax_online.argtypes = [P, I, I64, I64, P, P, P]
        lib.orc_md_merge.argtypes = [D, D, D, D, P, P]
        lib.orc_softmax_chunked_stats.argtypes = [P, I, I64, I64, I64, P, P]
        lib.orc_log_softmax.argtypes = [P, I, I64, I64, P]
        lib.orc_logsumexp_argmax.argtypes = [P, I, I64, I64, P, P]
        lib.orc_topk.argtypes = [P, I, I64, I64, I64, P, P, P, P]
        lib.orc_layernorm.argtypes = [P, P, P, I, D, I64, I64, P, P, P]
        lib.orc_welford.argtypes = [P, I, I64, I64, P, P, P]
        lib.orc_chan_merge.argtypes = [D, D, D, D, D, D, P, P, P]
        return lib


def _load():
    global _lib
    with _lock:
        if _lib is None:
            _lib = _configure(ctypes.CDLL(build()))
        return _lib


def compile_variant(src_text: str, out_path: str) -> str:
    """Compile a modified copy of oracle.c (used by the pin-strength tests,
    which plant mistakes in a copy and check that the pins catch them)."""
    src = out_path[:-3] + ".c"
    with open(src, "w") as f:
        f.write(src_text)
    subprocess.run(["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-fopenmp", src, "-o", out_path,
                    "-lm"], check=True)
    return out_path


class use_library:
    """Context manager: route every oracle call to the library at `path`."""

    def __init__(self, path: str):
        self.path = path

    def __enter__(self):
        global _lib
        _load()
        with _lock:
            self.saved = _lib
            _lib = _configure(ctypes.CDLL(self.path))
        return self

    def __exit__(self, *exc):
        global _lib
        with _lock:
            _lib = self.saved


def _dt(a: np.ndarray) -> int:
    if a.dtype == np.float32:
        return F32
    if a.dtype == np.uint16:
        return BF16
    raise TypeError(f"oracle inputs are float32 or uint16 (bfloat16 bits), got {a.dtype}")


def _c(a: np.ndarray) -> np.ndarray:
    return np.ascontiguousarray(a)


def _ptr(a: np.ndarray):
    return a.ctypes.data_as(ctypes.c_void_p)


def _rows(a: np.ndarray):
    if a.ndim == 1:
        return 1, a.shape[0]
    if a.ndim != 2:
        raise ValueError("rows are given as a 1-D or 2-D array")
    return a.shape


def set_threads(n: int) -> None:
    _load().orc_set_threads(int(n))


def get_threads() -> int:
    return int(_load().orc_get_threads())


def round_bf16_bits(v: float) -> int:
    """Bit pattern of the bfloat16 nearest to v (ties to even), rounded once."""
    return int(_load().orc_round_bf16(float(v)))


def round_to(v: np.ndarray, dtype: str) -> np.ndarray:
    """Round float64 values once to 'f32' (float32 array) or 'bf16' (uint16 bits)."""
    v = _c(np.asarray(v, dtype=np.float64))
    out = np.empty(v.shape, dtype=np.float32 if dtype == "f32" else np.uint16)
    _load().orc_round_array(_ptr(v), v.size, F32 if dtype == "f32" else BF16, _ptr(out))
    return out


def rmsnorm(x: np.ndarray, gamma: np.ndarray, eps: float, return_rstd: bool = False):
    x, gamma = _c(x), _c(gamma)
    dt = _dt(x)
    if _dt(gamma) != dt:
        raise TypeError("gamma has the storage type of x")
    M, H = _rows(x)
    y = np.empty((M, H), dtype=np.float64)
    r = np.empty(M, dtype=np.float64)
    _load().orc_rmsnorm(_ptr(x), _ptr(gamma), dt, float(eps), M, H, _ptr(y), _ptr(r))
    return (y, r) if return_rstd else y


def fused_add_rmsnorm(x: np.ndarray, residual: np.ndarray, gamma: np.ndarray, eps: float,
                      return_rstd: bool = False):
    """Returns (new_residual, out[, rstd]) as float64 arrays."""
    x, residual, gamma = _c(x), _c(residual), _c(gamma)
    dt = _dt(x)
    if _dt(residual) != dt or _dt(gamma) != dt:
        raise TypeError("x, residual and gamma share one storage type")
    M, H = _rows(x)
    h = np.empty((M, H), dtype=np.float64)
    y = np.empty((M, H), dtype=np.float64)
    r = np.empty(M, dtype=np.float64)
    _load().orc_fused_add_rmsnorm(_ptr(x), _ptr(residual), _ptr(gamma), dt, float(eps), M, H,
                                  _ptr(h), _ptr(y), _ptr(r))
    return (h, y, r) if return_rstd else (h, y)


def softmax(x: np.ndarray, return_stats: bool = False):
    """Three-pass safe softmax in binary64; stats are (m, d) per row."""
    x = _c(x)
    M, N = _rows(x)
    y = np.empty((M, N), dtype=np.float64)
    m = np.empty(M, dtype=np.float64)
    d = np.empty(M, dtype=np.float64)
    _load().orc_softmax(_ptr(x), _dt(x), M, N, _ptr(y), _ptr(m), _ptr(d))
    return (y, m, d) if return_stats else y


def softmax_online(x: np.ndarray, return_stats: bool = False):
    """Element-at-a-time online normaliser in binary64 (non-empty finite rows)."""
    x = _c(x)
    M, N = _rows(x)
    y = np.empty((M, N), dtype=np.float64)
    m = np.empty(M, dtype=np.float64)
    d = np.empty(M, dtype=np.float64)
    _load().orc_softmax_online(_ptr(x), _dt(x), M, N, _ptr(y), _ptr(m), _ptr(d))
    return (y, m, d) if return_stats else y


def md_merge(a, b):
    """(m1, d1) (+) (m2, d2) in binary64."""
    m = ctypes.c_double()
    d = ctypes.c_double()
    _load().orc_md_merge(float(a[0]), float(a[1]), float(b[0]), float(b[1]),
                         ctypes.byref(m), ctypes.byref(d))
    return (m.value, d.value)


def softmax_chunked_stats(x: np.ndarray, chunk: int):
    x = _c(x)
    M, N = _rows(x)
    m = np.empty(M, dtype=np.float64)
    d = np.empty(M, dtype=np.float64)
    _load().orc_softmax_chunked_stats(_ptr(x), _dt(x), M, N, int(chunk), _ptr(m), _ptr(d))
    return m, d


def log_softmax(x: np.ndarray):
    """log softmax in binary64, as (x - m) - log d."""
    x = _c(x)
    M, N = _rows(x)
    y = np.empty((M, N), dtype=np.float64)
    _load().orc_log_softmax(_ptr(x), _dt(x), M, N, _ptr(y))
    return y


def logsumexp_argmax(x: np.ndarray):
    """Per row: (m + log d) as float64 and the first index of the maximum."""
    x = _c(x)
    M, N = _rows(x)
    lse = np.empty(M, dtype=np.float64)
    am = np.empty(M, dtype=np.int64)
    _load().orc_logsumexp_argmax(_ptr(x), _dt(x), M, N, _ptr(lse), _ptr(am))
    return lse, am


def topk(x: np.ndarray, k: int):
    """Per row, the k largest values in the top-k order (value descending,
    equal values by lower index, NaN above every number), their column
    indices, the softmax of those k values and the row's log-sum-exp.
    Returns (values float64 [M, k], indices int64 [M, k], probs float64
    [M, k], lse float64 [M])."""
    x = _c(x)
    M, N = _rows(x)
    if not 1 <= k <= N:
        raise ValueError("need 1 <= k <= N")
    vals = np.empty((M, k), dtype=np.float64)
    idx = np.empty((M, k), dtype=np.int64)
    probs = np.empty((M, k), dtype=np.float64)
    lse = np.empty(M, dtype=np.float64)
    _load().orc_topk(_ptr(x), _dt(x), M, N, int(k), _ptr(vals), _ptr(idx), _ptr(probs), _ptr(lse))
    return vals, idx, probs, lse


def layernorm(x: np.ndarray, gamma: np.ndarray, beta: np.ndarray, eps: float,
              return_stats: bool = False):
    """Two-pass LayerNorm in binary64; stats are (mean, rstd) per row."""
    x, gamma, beta = _c(x), _c(gamma), _c(beta)
    dt = _dt(x)
    if _dt(gamma) != dt or _dt(beta) != dt:
        raise TypeError("x, gamma and beta share one storage type")
    M, H = _rows(x)
    y = np.empty((M, H), dtype=np.float64)
    mu = np.empty(M, dtype=np.float64)
    r = np.empty(M, dtype=np.float64)
    _load().orc_layernorm(_ptr(x), _ptr(gamma), _ptr(beta), dt, float(eps), M, H, _ptr(y), _ptr(mu),
                          _ptr(r))
    return (y, mu, r) if return_stats else y


def welford(x: np.ndarray):
    """Welford's (n, mean, M2) of each row, one element at a time."""
    x = _c(x)
    M, N = _rows(x)
    n, mu, m2 = (np.empty(M, dtype=np.float64) for _ in range(3))
    _load().orc_welford(_ptr(x), _dt(x), M, N, _ptr(n), _ptr(mu), _ptr(m2))
    return n, mu, m2


def chan_merge(a, b):
    """Chan's merge of two (n, mean, M2) states."""
    out = [ctypes.c_double() for _ in range(3)]
    _load().orc_chan_merge(*(float(v) for v in a), *(float(v) for v in b),
                           *(ctypes.byref(o) for o in out))
    return tuple(o.value for o in out)
