"""Seeded random shapes through every operation, against the fp64 oracle.

Row counts, row lengths (log-uniform up to 70 K elements), dtypes, a
one-element misalignment and the in-place form are drawn per case, so the
dispatcher's tier boundaries and ragged tails are crossed at sizes no
hand-picked list names.  Tolerances are those of the other parity tests."""
import random

import numpy as np
import pytest
import torch

import oracle
import online_softmax_row_gb300 as osr
import workloads
from parity import check_bf16, check_f32_abs, check_out, check_row_max_and_argmax, seed_of, to_oracle_input
from test_gpu_layernorm import EPS as LN_EPS, check_ln  # LayerNorm's own tolerance check

pytestmark = pytest.mark.gpu

DT = {"f32": torch.float32, "bf16": torch.bfloat16}
CASES = 40


@pytest.fixture(scope="module", autouse=True)
def gpu():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    osr.library()


def draw(op, i):
    rnd = random.Random(seed_of("random-shapes", op, i))
    N = max(1, int(round(10 ** rnd.uniform(0, np.log10(70000)))))
    M = max(1, min(rnd.choice([1, 2, 3, 7, 16, 37, 64, 150, 300]), (4 << 20) // N))
    dt = rnd.choice(["f32", "bf16"])
    odt = rnd.choice(["f32", "bf16"])
    shift = rnd.random() < 0.3
    in_place = rnd.random() < 0.25
    return M, N, dt, odt, shift, in_place


def on_device(t: torch.Tensor, shift: bool) -> torch.Tensor:
    """t on the GPU, one element past a 16-byte boundary when shift."""
    if not shift:
        return t.cuda()
    buf = torch.empty(t.numel() + 1, dtype=t.dtype, device="cuda")
    v = buf[1:].view(t.shape)
    v.copy_(t)
    return v


@pytest.mark.parametrize("i", range(CASES))
def test_random_softmax_family(i):
    M, N, dt, odt, shift, in_place = draw("softmax", i)
    x = workloads.softmax_inputs(M, N, dt, sigma=4.0, shift_rows=M // 4, seed=seed_of("rs-x", i))["x"]
    xo = to_oracle_input(x)
    ref, m_ref, d_ref = oracle.softmax(xo, return_stats=True)
    what = f"softmax {M}x{N} {dt}->{odt} shift={shift} in_place={in_place}"
    xd = on_device(x, shift)
    if in_place:
        y = osr.softmax_rows(xd, out=xd)
        check_out(y, ref, what)
    else:
        y, rmax, rsum = osr.softmax_rows_stats(xd, out_dtype=DT[odt])
        torch.cuda.synchronize()
        check_out(y, ref, what)
        check_row_max_and_argmax(xo, y, rmax, m_ref, what)
        assert np.all(np.abs(rsum.cpu().numpy().astype(np.float64) - d_ref) <= 1e-5 * d_ref), what
    xd = on_device(x, shift)
    ly = osr.log_softmax_rows(xd, out_dtype=DT[odt])
    torch.cuda.synchronize()
    lref = oracle.log_softmax(xo)
    if odt == "f32":
        check_f32_abs(ly, lref, 4e-6, 1e-5, "log-" + what)
    else:
        check_bf16(ly, lref, "log-" + what, atol=4e-6, rtol=1e-5)
    lse, am = osr.row_logsumexp(on_device(x, shift))
    torch.cuda.synchronize()
    r_lse, r_am = oracle.logsumexp_argmax(xo)
    assert np.array_equal(am.cpu().numpy(), r_am), "argmax " + what
    check_f32_abs(lse, r_lse, 4e-6, 2e-7, "lse " + what)


@pytest.mark.parametrize("i", range(CASES))
def test_random_norms(i):
    M, N, dt, _, shift, in_place = draw("norms", i)
    eps = 1e-6
    inp = workloads.rmsnorm_inputs(M, N, dt, fused=True, seed=seed_of("rs-n", i))
    xo, go = to_oracle_input(inp["x"]), to_oracle_input(inp["gamma"])
    what = f"norms {M}x{N} {dt} shift={shift} in_place={in_place}"
    xd, gd = on_device(inp["x"], shift), on_device(inp["gamma"], shift)
    y = osr.rmsnorm_fwd(xd, gd, eps, out=xd if in_place else None)
    torch.cuda.synchronize()
    check_out(y, oracle.rmsnorm(xo, go, eps), "rmsnorm " + what)
    xd = on_device(inp["x"], shift)
    res = on_device(inp["residual"], shift)
    out = osr.fused_add_rmsnorm(xd, res, gd, eps, out=xd if in_place else None)
    torch.cuda.synchronize()
    h_ref, y_ref = oracle.fused_add_rmsnorm(xo, to_oracle_input(inp["residual"]), go, eps)
    if dt == "f32":
        assert np.array_equal(res.cpu().numpy().astype(np.float64), h_ref), "residual " + what
    else:
        check_bf16(res, h_ref, "residual " + what)
    check_out(out, y_ref, "fused " + what)
    beta = torch.randn(N, generator=torch.Generator().manual_seed(seed_of("rs-b", i))).to(DT[dt])
    xd = on_device(inp["x"], shift)
    ln = osr.layernorm_fwd(xd, gd, on_device(beta, shift), LN_EPS, out=xd if in_place else None)
    torch.cuda.synchronize()
    check_ln(inp["x"], inp["gamma"], beta, ln)


@pytest.mark.parametrize("i", range(CASES // 2))
def test_random_topk(i):
    M, N, dt, _, shift, _ = draw("topk", i)
    k = max(1, min(N, random.Random(seed_of("rs-k", i)).choice([1, 5, 50, 256, 1024])))
    x = workloads.softmax_inputs(M, N, dt, sigma=4.0, seed=seed_of("rs-t", i))["x"]
    xo = to_oracle_input(x)
    r_v, r_i, r_p, r_l = oracle.topk(xo, k)
    v, idx, p, lse = osr.row_topk(on_device(x, shift), k)
    torch.cuda.synchronize()
    what = f"topk {M}x{N} k={k} {dt} shift={shift}"
    assert np.array_equal(idx.cpu().numpy(), r_i), what
    assert np.array_equal(v.cpu().numpy().astype(np.float64), r_v), what
    check_f32_abs(p, r_p, 1e-6, 1e-5, "probs " + what)
    check_f32_abs(lse, r_l, 4e-6, 2e-7, "lse " + what)
