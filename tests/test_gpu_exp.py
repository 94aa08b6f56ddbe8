"""The kernels' exponential against its error bound and CUDA's expf.

Every softmax kernel takes e^(x - m) as ex2.approx.ftz.f32 applied to
p = fl(fl(x - m) * L), L = log2(e) rounded to binary32 (the identity
e^t = 2^(t log2 e)).  With t = x - m:
  p = t log2(e) (1 + d1)(1 + dL)(1 + d2),  |d1|, |d2| <= 2^-24, |dL| <= 2^-25,
so 2^p = e^t e^(t (d1 + dL + d2)), a relative error of at most
2.5 |t| 2^-24 (first order), and the special-function instruction adds at
most 2 ulp (2^-22 relative).  Bound tested, for results in the normal range
(e^t >= 2^-126):
  |approx - e^t| <= e^t (2^-22 + 2.5 |t| 2^-24) (1 + 2^-10)
Below the normal range the result flushes to 0 (or rounds to 2^-126).  The
bound stays within the softmax tolerance (1e-5 relative) for t >= -66, i.e.
for every output above e^-66 of the row's largest; it reaches 1.3e-5 at the
last normal result (t = -87.3).  CUDA's expf, given the rounded difference
fl(x - m), must be within its own 2 ulp (2^-22 relative) of e^fl(x - m), which
checks the harness."""
import ctypes

import numpy as np
import pytest
import torch

import online_softmax_row_gb300 as osr

pytestmark = pytest.mark.gpu
FLT_MIN = 2.0 ** -126


@pytest.fixture(scope="module")
def exp_shifted():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    fn = osr.library().osr_test_exp_shifted
    fn.argtypes = [ctypes.c_void_p] * 4 + [ctypes.c_int64, ctypes.c_void_p]
    fn.restype = ctypes.c_int

    def run(x: np.ndarray, m: np.ndarray):
        xd = torch.from_numpy(x.astype(np.float32)).cuda()
        md = torch.from_numpy(m.astype(np.float32)).cuda()
        a, r = torch.empty_like(xd), torch.empty_like(xd)
        assert fn(xd.data_ptr(), md.data_ptr(), a.data_ptr(), r.data_ptr(), xd.numel(),
                  torch.cuda.current_stream().cuda_stream) == 0
        torch.cuda.synchronize()
        return a.cpu().numpy().astype(np.float64), r.cpu().numpy().astype(np.float64)
    return run


def _inputs():
    rng = np.random.default_rng(20240)
    ts = np.concatenate([-np.linspace(0.0, 104.0, 1 << 20), -rng.uniform(0, 104, 1 << 20),
                         -rng.exponential(2.0, 1 << 18)])
    xs, ms = [], []
    for m in (0.0, 3.5, 30.0, -40.0, 1000.0, 12.345678):
        m32 = np.float32(m)
        xs.append((np.float64(m32) + ts).astype(np.float32))
        ms.append(np.full(ts.size, m32, dtype=np.float32))
    # softmax-like pairs: x ~ N(0, 16), m the largest of a few thousand draws
    x = (rng.standard_normal(1 << 20) * 4).astype(np.float32)
    xs.append(x)
    ms.append(np.full(x.size, np.float32(x.max()), dtype=np.float32))
    return np.concatenate(xs), np.concatenate(ms)


def test_exp_shifted_within_its_bound(exp_shifted):
    x, m = _inputs()
    approx, ref = exp_shifted(x, m)
    t = x.astype(np.float64) - m.astype(np.float64)
    truth = np.exp(t)
    normal = truth >= FLT_MIN
    rel = np.abs(approx[normal] - truth[normal]) / truth[normal]
    bound = (2.0 ** -22 + 2.5 * np.abs(t[normal]) * 2.0 ** -24) * (1 + 2.0 ** -10)
    worst = np.argmax(rel - bound)
    assert np.all(rel <= bound), (f"t={t[normal][worst]!r}: relative error {rel[worst]:.3g} "
                                  f"above the bound {bound[worst]:.3g}")
    near = np.abs(t[normal]) <= 66.0
    assert rel[near].max() <= 1e-5
    tiny = ~normal
    assert np.all((approx[tiny] >= 0) & (approx[tiny] <= FLT_MIN * (1 + 2.0 ** -20)))
    # CUDA's expf of the rounded difference fl(x - m) (what it is given),
    # within its 2 ulp of e^fl(x - m)
    t32 = (x - m).astype(np.float64)  # binary32 subtraction, rounded as on the device
    truth32 = np.exp(t32)
    n32 = truth32 >= FLT_MIN
    ref_rel = np.abs(ref[n32] - truth32[n32]) / truth32[n32]
    assert ref_rel.max() <= 2.0 ** -22


def test_exp_shifted_special_values(exp_shifted):
    inf, nan = np.inf, np.nan
    x = np.array([-inf, -inf, 5.0, nan, 0.0, -1e30, 7.0, -104.0], dtype=np.float32)
    m = np.array([0.0, 10.0, 5.0, 0.0, -0.0, 0.0, 7.0, 0.0], dtype=np.float32)
    a, _ = exp_shifted(x, m)
    assert a[0] == 0.0 and a[1] == 0.0       # e^-inf = 0: masked entries
    assert a[2] == 1.0 and a[6] == 1.0       # the row maximum itself: exactly 1
    assert np.isnan(a[3])                    # NaN propagates
    assert a[4] == 1.0
    assert a[5] == 0.0 and a[7] == 0.0       # far below the normal range: flushed
