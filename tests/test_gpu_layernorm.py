"""LayerNorm through the C ABI against the fp64 oracle.

Tolerance, derived from the binary32 arithmetic: y = z * gamma + beta with
z = ((x - p) - mu_s) * r; the summation trees for mu_s and var put a relative
error of a few 1e-6 into z, and the final addition of beta can cancel, so the
error is bounded by the size of the terms, not of the result:
  binary32 out: |gpu - ref| <= 1e-6 + 1e-5 (|z gamma| + |beta|)
  bf16 out:     |gpu - ref| <= one bf16 ulp of ref + 1e-6 + 1e-5 (|z gamma| + |beta|)
with z, gamma, beta from the oracle's statistics (fp64).  The 1e-6 is the
binary32 arithmetic's absolute floor for both output types: the mean's
summation tree rounds at the scale of sum(x - p), and an output that cancels
to near zero (z gamma = -beta, both small) keeps that absolute error."""
import os

import numpy as np
import pytest
import torch

import oracle
import online_softmax_row_gb300 as osr
import workloads
from parity import seed_of, bits16, to_oracle_input

pytestmark = pytest.mark.gpu
EPS = 1e-5


@pytest.fixture(scope="module", autouse=True)
def gpu():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    osr.library()



def ln_case(M, H, dt, seed, lo=None, hi=None):
    g = torch.Generator().manual_seed(seed)
    if lo is None:
        x = torch.randn(M, H, generator=g)
    else:
        x = torch.rand(M, H, generator=g) * (hi - lo) + lo
    gamma = torch.rand(H, generator=g) + 0.5
    beta = torch.randn(H, generator=g)
    t = {"f32": torch.float32, "bf16": torch.bfloat16}[dt]
    return x.to(t), gamma.to(t), beta.to(t)


def f64(t):
    t = t.detach().cpu()
    return t.double().numpy()


def check_ln(x, gamma, beta, y):
    xo, go, bo = (to_oracle_input(t) for t in (x, gamma, beta))
    ref, mu, r = oracle.layernorm(xo.reshape(y.shape[0], -1), go, bo, EPS, return_stats=True)
    ref = ref.reshape(y.shape)
    z = (f64(x).reshape(ref.shape) - mu[:, None]) * r[:, None]
    scale = np.abs(z * f64(gamma)) + np.abs(f64(beta))
    got = f64(y).reshape(ref.shape)
    if y.dtype == torch.float32:
        bound = 1e-6 + 1e-5 * scale
    else:
        ulp = np.where(ref != 0, 2.0 ** (np.floor(np.log2(np.abs(ref) + 1e-300)) - 7), 2.0 ** -133)
        bound = ulp + 1e-6 + 1e-5 * scale
    bad = ~(np.abs(got - ref) <= bound)
    if bad.any():
        i = tuple(np.argwhere(bad)[0])
        raise AssertionError(f"layernorm: {bad.sum()} outside tolerance, first {i}: gpu={got[i]} ref={ref[i]}")


SHAPES = [(1, 1), (7, 2), (5, 3), (4, 33), (9, 128), (33, 1000), (3, 1023), (64, 3584),
          (4, 4096), (2, 4097), (3, 16384), (2, 32768), (2, 50000), (2, 300000)]


@pytest.mark.parametrize("dt", ["f32", "bf16"])
@pytest.mark.parametrize("M,H", SHAPES)
def test_layernorm(M, H, dt):
    x, g, b = ln_case(M, H, dt, seed_of("ln", M, H, dt))
    y = osr.layernorm_fwd(x.cuda(), g.cuda(), b.cuda(), EPS)
    torch.cuda.synchronize()
    check_ln(x, g, b, y)


@pytest.mark.parametrize("dt", ["f32", "bf16"])
def test_layernorm_mean_101_stress(dt):
    # rows in U(100, 102): mean ~101, standard deviation ~0.58, as in the
    # pages' LayerNorm exercise (256 x 5120); E[x^2] - E[x]^2 would lose it
    x, g, b = ln_case(256, 5120, dt, 7, 100.0, 102.0)
    y = osr.layernorm_fwd(x.cuda(), g.cuda(), b.cuda(), EPS)
    torch.cuda.synchronize()
    check_ln(x, g, b, y)


@pytest.mark.parametrize("spec", ["rows:g=512", "rows:g=1024", "cluster:g=256,cs=2",
                                  "cluster:g=256,cs=5", "cluster:g=1024,cs=1", "cluster:g=1024,cs=3",
                                  "split:s=1,b=64", "split:s=3,b=5", "split:s=7,b=37",
                                  "split:s=40,b=2"])
@pytest.mark.parametrize("dt", ["f32", "bf16"])
def test_layernorm_every_tier(spec, dt):
    x, g, b = ln_case(37, 5000, dt, seed_of("lnt", spec, dt), 100.0, 102.0)
    with osr.forced_kernel(spec):
        y = osr.layernorm_fwd(x.cuda(), g.cuda(), b.cuda(), EPS)
        torch.cuda.synchronize()
    check_ln(x, g, b, y)


@pytest.mark.parametrize("spec", [None, "cluster:g=256,cs=4", "split:s=9,b=2"])
def test_layernorm_in_place_and_misaligned(spec):
    x, g, b = ln_case(6, 4001, "f32", seed_of("lnip", spec), -3.0, 5.0)
    buf = torch.empty(6 * 4001 + 1, device="cuda")
    xm = buf[1:].view(6, 4001)
    xm.copy_(x.cuda())
    with osr.forced_kernel(spec):
        osr.layernorm_fwd(xm, g.cuda(), b.cuda(), EPS, out=xm)
        torch.cuda.synchronize()
    check_ln(x, g, b, xm)
    # aligned, in place, through every tier
    x2, g2, b2 = ln_case(5, 8192, "bf16", seed_of("lnip2", spec))
    xc = x2.cuda()
    with osr.forced_kernel(spec):
        osr.layernorm_fwd(xc, g2.cuda(), b2.cuda(), EPS, out=xc)
        torch.cuda.synchronize()
    check_ln(x2, g2, b2, xc)


def test_layernorm_constant_rows_give_beta():
    x = torch.full((3, 1000), 101.25, device="cuda")
    g = torch.rand(1000, device="cuda") + 0.5
    b = torch.randn(1000, device="cuda")
    y = osr.layernorm_fwd(x, g, b, EPS)
    assert torch.equal(y, b.expand(3, -1))


def test_layernorm_workloads_full_size():
    for name in ("layernorm_f32_256x5120_mean101", "layernorm_bf16_8192x4096"):
        w = workloads.WORKLOADS[name]
        inp = workloads.make(w)
        y = osr.layernorm_fwd(inp["x"].cuda(), inp["gamma"].cuda(), inp["beta"].cuda(), w.eps)
        torch.cuda.synchronize()
        check_ln(inp["x"], inp["gamma"], inp["beta"], y)


def test_layernorm_on_pinned_host_rows():
    import ctypes
    lib = osr.library()
    inp = workloads.layernorm_inputs(16, 5120, "f32", low=100.0, high=102.0, seed=31)
    hx, hg, hb = (inp[k].clone().pin_memory() for k in ("x", "gamma", "beta"))
    hy = torch.empty_like(hx).pin_memory()
    st = torch.cuda.current_stream().cuda_stream
    assert lib.osr_layernorm_fwd(hx.data_ptr(), hg.data_ptr(), hb.data_ptr(), ctypes.c_float(1e-5),
                                 hy.data_ptr(), 16, 5120, 0, st) == 0
    torch.cuda.synchronize()
    dy = osr.layernorm_fwd(inp["x"].cuda(), inp["gamma"].cuda(), inp["beta"].cuda(), 1e-5)
    torch.cuda.synchronize()
    assert torch.equal(hy, dy.cpu())


@pytest.mark.parametrize("H", [4096, 5120, 65536])
def test_layernorm_bf16_one_pass_and_far_pivot(H):
    # bf16 rows take their statistics in one pass about the pivot x[row][0];
    # a pivot far from the mean (rows 0-1: x[0] = +-300 in N(0,1) rows) or an
    # offset mean (rows 2-3: N(100, 1), N(-1000, 4)) loses digits there, and
    # the exact second pass about the mean must take over
    x, gamma, beta = ln_case(6, H, "f32", seed_of("ln-pivot", H))
    x = x.float()
    x[0, 0] = 300.0
    x[1, 0] = -300.0
    x[2] = x[2] + 100.0
    x[3] = x[3] * 4.0 - 1000.0
    xb, gb, bb = x.to(torch.bfloat16), gamma.to(torch.bfloat16), beta.to(torch.bfloat16)
    y = osr.layernorm_fwd(xb.cuda(), gb.cuda(), bb.cuda(), EPS)
    torch.cuda.synchronize()
    check_ln(xb, gb, bb, y.cpu())
