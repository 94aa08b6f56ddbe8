"""Element-by-element comparison of CUDA results with the fp64 oracle.

Tolerances (from the stated targets):
  binary32 outputs: |gpu - ref| <= 1e-6 + 1e-5 |ref| for every element, and
                    |gpu - ref| / |ref| <= 1e-5 wherever ref is a normal
                    binary32 number (|ref| >= 2^-126);
  bfloat16 outputs: within 1 bf16 ulp of the oracle's value rounded once to
                    bf16 (ordered-integer distance of the bit patterns);
  row max:          bit-exact; the position of the oracle's argmax holds the
                    row's largest GPU output.
"""
import zlib

import numpy as np
import torch

import oracle


def seed_of(*k) -> int:
    """A stable seed from a test's parameters (the same in every process)."""
    return zlib.crc32(repr(k).encode()) & 0x7FFFFFFF

ATOL, RTOL = 1e-6, 1e-5
FLT_MIN = 2.0 ** -126


def bits16(t: torch.Tensor) -> np.ndarray:
    return t.detach().contiguous().cpu().view(torch.int16).numpy().view(np.uint16)


def to_oracle_input(t: torch.Tensor) -> np.ndarray:
    """float32 array, or uint16 bit patterns for bfloat16, as the oracle takes."""
    t = t.detach().contiguous().cpu()
    if t.dtype == torch.bfloat16:
        return t.view(torch.int16).numpy().view(np.uint16)
    return t.numpy()


def _ordered16(b: np.ndarray) -> np.ndarray:
    b = b.astype(np.int64)
    return np.where(b & 0x8000, 0x8000 - (b & 0x7FFF), 0x8000 + b)


def check_f32(got: torch.Tensor, ref: np.ndarray, what: str = ""):
    g = got.detach().cpu().numpy().astype(np.float64).reshape(ref.shape)
    both_nan = np.isnan(g) & np.isnan(ref)
    err = np.abs(g - ref)
    bad = ~both_nan & ~(err <= ATOL + RTOL * np.abs(ref))
    if bad.any():
        i = np.argwhere(bad)[0]
        raise AssertionError(f"{what}: {bad.sum()} elements outside atol/rtol; first at {tuple(i)}: "
                             f"gpu={g[tuple(i)]!r} ref={ref[tuple(i)]!r}")
    normal = ~both_nan & (np.abs(ref) >= FLT_MIN)
    if normal.any():
        rel = (err[normal] / np.abs(ref[normal])).max()
        assert rel <= RTOL, f"{what}: max relative error {rel:.3g} > {RTOL}"
        return float(rel)
    return 0.0


def check_f32_abs(got: torch.Tensor, ref: np.ndarray, atol: float, rtol: float, what: str = ""):
    """|gpu - ref| <= atol + rtol |ref| for every element (NaN matches NaN,
    equal infinities match)."""
    g = got.detach().cpu().numpy().astype(np.float64).reshape(ref.shape)
    same = (np.isnan(g) & np.isnan(ref)) | (g == ref)
    err = np.abs(g - ref)
    bad = ~same & ~(err <= atol + rtol * np.abs(ref))
    if bad.any():
        i = np.argwhere(bad)[0]
        raise AssertionError(f"{what}: {bad.sum()} elements outside tolerance; first at {tuple(i)}: "
                             f"gpu={g[tuple(i)]!r} ref={ref[tuple(i)]!r}")


def check_bf16(got: torch.Tensor, ref: np.ndarray, what: str = "", max_ulp: int = 1,
               atol: float = 0.0, rtol: float = 0.0):
    """Within max_ulp bf16 ulp of the oracle rounded once to bf16; with atol
    or rtol given, an element may instead lie within atol + rtol |ref| plus
    one bf16 spacing of ref (for outputs whose binary32 error is absolute,
    such as log-softmax values near 0)."""
    g = bits16(got).reshape(ref.shape)
    r = oracle.round_to(ref, "bf16")
    nan = np.isnan(ref)
    gnan = (g & 0x7FFF) > 0x7F80
    assert np.array_equal(nan, gnan), f"{what}: NaN positions differ"
    d = np.abs(_ordered16(g[~nan]) - _ordered16(r[~nan]))
    bad = d > max_ulp
    if (atol or rtol) and bad.any():
        gv = (g[~nan].astype(np.uint32) << 16).view(np.float32).astype(np.float64)
        rv = ref[~nan]
        spacing = np.where(rv != 0, 2.0 ** (np.floor(np.log2(np.abs(rv) + 1e-300)) - 7), 2.0 ** -133)
        bad &= ~(np.abs(gv - rv) <= atol + rtol * np.abs(rv) + spacing)
    if bad.any():
        i = np.argmax(np.where(bad, d, -1))
        raise AssertionError(f"{what}: {int(bad.sum())} elements beyond {max_ulp} bf16 ulp; "
                             f"worst {int(d[i])} ulp")
    return int(d.max()) if d.size else 0


def check_out(got: torch.Tensor, ref: np.ndarray, what: str = ""):
    if got.dtype == torch.float32:
        return check_f32(got, ref, what)
    return check_bf16(got, ref, what)


def check_row_max_and_argmax(x_in: np.ndarray, y_gpu: torch.Tensor, row_max: torch.Tensor,
                             m_ref: np.ndarray, what: str = ""):
    gm = row_max.detach().cpu().numpy().astype(np.float64)
    assert np.array_equal(gm, m_ref), f"{what}: row max differs from the oracle's"
    y = y_gpu.detach().float().cpu().numpy()
    xs = x_in if x_in.dtype == np.float32 else (x_in.astype(np.uint32) << 16).view(np.float32)
    am = np.argmax(xs, axis=1)  # lowest index on ties
    got_at = y[np.arange(y.shape[0]), am]
    assert np.array_equal(got_at, y.max(axis=1)), f"{what}: argmax position is not the largest output"
