"""Degenerate rows through every dispatcher tier, against the fp64 oracle.

Each batch holds rows that are all -inf, have one finite entry (at a random
column, the first or the last), are -inf-heavy, hold +inf or NaN, are all
NaN, mix only -inf and NaN, have the dtype's lowest finite number as their
maximum, or are constant.  "GPU Kernel 工程（04）" 十.3 and 十.4 ask for exactly
these boundary rows; the identity (-inf, 0) is that of "两个融合算子" §5·三.

What is compared, per the header's stated semantics:
  row max      bit-exact with the oracle's m (NaN entries are skipped by the
               maximum; a row with no number above -inf has m = -inf);
  row sum      0 for a row of only -inf (the empty sum: every term is
               e^-inf; the oracle's exp(-inf - (-inf)) is undefined there),
               NaN where the oracle's d is NaN, else within 1e-5 relative;
  softmax      element by element with the oracle (NaN rows match NaN);
  log-softmax  element by element with the oracle (equal infinities match);
  lse/argmax   a row of only -inf gives lse = -inf and argmax = -1, every
               other row the oracle's values;
  top-k        values and indices bit-exact, probs and lse as above.
"""
import os

import numpy as np
import pytest
import torch

import oracle
import online_softmax_row_gb300 as osr
from parity import check_bf16, check_f32_abs, check_out, seed_of, to_oracle_input

pytestmark = pytest.mark.gpu

DT = {"f32": torch.float32, "bf16": torch.bfloat16}
ROWS = 12


@pytest.fixture(scope="module", autouse=True)
def gpu():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    osr.library()


def degenerate_rows(N: int, dt: str, seed: int) -> torch.Tensor:
    g = torch.Generator().manual_seed(seed)
    base = torch.randn(ROWS, N, generator=g) * 4.0
    cols = torch.randint(0, N, (ROWS,), generator=g).tolist()
    x = base.clone()
    inf, nan = float("inf"), float("nan")
    x[0] = -inf                                            # all -inf
    x[1] = -inf
    x[1, cols[1]] = base[1, cols[1]]                       # one finite entry
    x[2][torch.rand(N, generator=g) < 0.95] = -inf         # -inf-heavy
    x[3, cols[3]] = inf                                    # one +inf
    x[4, cols[4]] = nan                                    # one NaN
    x[6] = nan                                             # all NaN
    x[7] = -inf
    x[7][torch.rand(N, generator=g) < 0.5] = nan           # only -inf and NaN
    x[8] = -inf
    x[8, 0] = base[8, 0]                                   # finite entry first
    x[9] = -inf
    x[9, N - 1] = base[9, N - 1]                           # finite entry last
    x[10] = -inf
    x[10, cols[10]] = torch.finfo(DT[dt]).min              # lowest finite max
    x[10, (cols[10] + N // 2) % N] = torch.finfo(DT[dt]).min
    x[11] = 5.0                                            # constant
    return x.to(DT[dt])


def run_forced(spec, fn):
    with osr.forced_kernel(spec):
        out = fn()
        torch.cuda.synchronize()
        return out


def all_minus_inf(xo: np.ndarray) -> np.ndarray:
    xs = xo if xo.dtype == np.float32 else (xo.astype(np.uint32) << 16).view(np.float32)
    return np.all(xs == -np.inf, axis=1)


def check_stats(xo, rmax, rsum, m_ref, d_ref, what):
    gm = rmax.cpu().numpy().astype(np.float64)
    assert np.array_equal(gm, m_ref), f"{what}: row max {gm} vs oracle {m_ref}"
    gd = rsum.cpu().numpy().astype(np.float64)
    empty = all_minus_inf(xo)
    assert np.all(gd[empty] == 0.0), f"{what}: row sum of a row of only -inf is {gd[empty]}"
    nan = np.isnan(d_ref) & ~empty
    assert np.all(np.isnan(gd[nan])), f"{what}: row sum should be NaN where the oracle's is"
    fin = ~nan & ~empty
    assert np.all(np.abs(gd[fin] - d_ref[fin]) <= 1e-5 * d_ref[fin]), f"{what}: row sum"


# (forced plan, row length): every softmax tier, the element-wise path, and
# the default plan of a vocabulary row (staged)
SOFTMAX_TIERS = [("rows:g=4", 64), ("rows:g=32", 504), ("rows:g=512", 5000), ("rows:g=512", 5001),
                 ("cluster:g=256,cs=3", 5000), ("cluster:g=1024,cs=2", 6000),
                 ("staged:cs=3,r=0", 5000), ("staged:cs=1,r=8", 5000), ("staged:cs=3,r=8", 40008),
                 ("staged:cs=16,r=0", 40000), ("split:s=1,b=64", 5000), ("split:s=5,b=4", 5000),
                 ("split:s=7,b=3", 5001), (None, 152064)]


@pytest.mark.parametrize("io", [("f32", "f32"), ("bf16", "f32"), ("bf16", "bf16"), ("f32", "bf16")])
@pytest.mark.parametrize("spec,N", SOFTMAX_TIERS)
def test_softmax_and_log_softmax_degenerate_rows(spec, N, io):
    x = degenerate_rows(N, io[0], seed_of("degen", spec, N, io))
    xo = to_oracle_input(x)
    ref, m_ref, d_ref = oracle.softmax(xo, return_stats=True)
    xd = x.cuda()
    y, rmax, rsum = run_forced(spec, lambda: osr.softmax_rows_stats(xd, out_dtype=DT[io[1]]))
    what = f"{spec or 'default'} N={N} {io}"
    check_stats(xo, rmax, rsum, m_ref, d_ref, what)
    check_out(y, ref, what)
    ly = run_forced(spec, lambda: osr.log_softmax_rows(xd, out_dtype=DT[io[1]]))
    lref = oracle.log_softmax(xo)
    if io[1] == "f32":
        check_f32_abs(ly, lref, 4e-6, 1e-5, f"log-softmax {what}")
    else:
        check_bf16(ly, lref, f"log-softmax {what}", atol=4e-6, rtol=1e-5)


@pytest.mark.parametrize("dt", ["f32", "bf16"])
@pytest.mark.parametrize("spec", ["rows:g=512", "cluster:g=256,cs=4", "staged:cs=5,r=0",
                                  "staged:cs=2,r=8", "split:s=6,b=5"])
def test_in_place_softmax_degenerate_rows(spec, dt):
    N = 40008 if spec.startswith("staged") else 5000
    x = degenerate_rows(N, dt, seed_of("degen-inplace", spec, dt))
    ref = oracle.softmax(to_oracle_input(x))
    xd = x.cuda()
    run_forced(spec, lambda: osr.softmax_rows(xd, out=xd))
    check_out(xd, ref, f"in place {spec} {dt}")


# log-sum-exp / argmax: short rows (groups of lanes), one CTA per row, the
# streaming cluster, the staged cluster, and narrow groups whose threads
# stream many tiles
LSE_TIERS = [(None, 64), (None, 5000), ("lse:cs=4,st=0", 152064), ("lse:cs=12,st=1", 152064),
             ("lse:cs=3,st=1", 40000), ("lse:cs=2,st=0", 5001),
             ("lse:g=1", 5000), ("lse:g=8", 4096),  # many tiles a thread
             ("lse:g=1024,cs=1", 40000)]            # one wide CTA a row


@pytest.mark.parametrize("dt", ["f32", "bf16"])
@pytest.mark.parametrize("spec,N", LSE_TIERS)
def test_logsumexp_argmax_degenerate_rows(spec, N, dt):
    x = degenerate_rows(N, dt, seed_of("degen-lse", spec, N, dt))
    xo = to_oracle_input(x)
    r_lse, r_am = oracle.logsumexp_argmax(xo)
    lse, am = run_forced(spec, lambda: osr.row_logsumexp(x.cuda()))
    lse, am = lse.cpu().numpy().astype(np.float64), am.cpu().numpy()
    empty = all_minus_inf(xo)
    assert np.all(lse[empty] == -np.inf) and np.all(am[empty] == -1), "rows of only -inf"
    assert np.array_equal(am[~empty], r_am[~empty]), f"argmax {am} vs {r_am}"
    check_f32_abs(torch.from_numpy(lse[~empty]), r_lse[~empty], 4e-6, 2e-7, f"lse {spec} N={N}")


@pytest.mark.parametrize("dt", ["f32", "bf16"])
@pytest.mark.parametrize("spec,N,k", [(None, 4096, 8), (None, 152064, 50), ("topk:cs=3", 40000, 50),
                                      (None, 3001, 16)])
def test_topk_degenerate_rows(spec, N, k, dt):
    x = degenerate_rows(N, dt, seed_of("degen-topk", spec, N, k, dt))
    xo = to_oracle_input(x)
    r_v, r_i, r_p, r_l = oracle.topk(xo, k)
    v, i, p, lse = run_forced(spec, lambda: osr.row_topk(x.cuda(), k))
    assert np.array_equal(i.cpu().numpy(), r_i), "top-k indices"
    gv = v.cpu().numpy().astype(np.float64)
    assert np.all((gv == r_v) | (np.isnan(gv) & np.isnan(r_v))), "top-k values"
    check_f32_abs(p, r_p, 1e-6, 1e-5, "top-k probs")
    empty = all_minus_inf(xo)
    gl = lse.cpu().numpy().astype(np.float64)
    assert np.all(gl[empty] == -np.inf), "top-k lse of rows of only -inf"
    check_f32_abs(torch.from_numpy(gl[~empty]), r_l[~empty], 4e-6, 2e-7, "top-k lse")
