"""Log-softmax and the per-row log-sum-exp / argmax against the fp64 oracle.

Tolerances derived from the binary32 arithmetic (the oracle is exact to
binary64):
  log-softmax, binary32 out: |gpu - ref| <= 4e-6 + 1e-5 |ref|.  The result is
    (x - m) - log d; d carries the rounding of its summation tree (at most
    ~2.5e-6 relative for the tiers here: 16 sequential terms per thread and
    <= 26 tree levels), which logf turns into an absolute error of the same
    size, plus one rounding each for x - m, log and the subtraction.  Values
    near 0 (a dominant row maximum) are bounded absolutely, not relatively.
  log-softmax, bf16 out: within 1 bf16 ulp, as for softmax, or, where the
    binary32 error is the absolute one above (values near 0: a dominant
    maximum gives -log d with d barely above 1), within 4e-6 + 1e-5 |ref|
    plus one bf16 spacing.
  log-sum-exp: |gpu - ref| <= 4e-6 + 2e-7 |ref| (the same d error, plus the
    rounding of m + log d to binary32).
  argmax: exact, the first index of the maximum on ties."""
import os

import numpy as np
import pytest
import torch

import oracle
import online_softmax_row_gb300 as osr
import workloads
from parity import seed_of, check_bf16, check_f32_abs, to_oracle_input

pytestmark = pytest.mark.gpu
DT = {"f32": torch.float32, "bf16": torch.bfloat16}


@pytest.fixture(scope="module", autouse=True)
def gpu():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    osr.library()



def case(M, N, dt, seed, sigma=4.0):
    return workloads.softmax_inputs(M, N, dt, sigma=sigma, shift_rows=M // 3, seed=seed)["x"]


def check_log(x_cpu, y):
    ref = oracle.log_softmax(to_oracle_input(x_cpu).reshape(y.shape[0], -1)).reshape(y.shape)
    if y.dtype == torch.float32:
        check_f32_abs(y, ref, 4e-6, 1e-5, "log-softmax")
    else:
        check_bf16(y, ref, "log-softmax", atol=4e-6, rtol=1e-5)


def check_lse(x_cpu, lse, am):
    xo = to_oracle_input(x_cpu).reshape(lse.shape[0], -1)
    r_lse, r_am = oracle.logsumexp_argmax(xo)
    assert np.array_equal(am.cpu().numpy(), r_am), "argmax"
    check_f32_abs(lse, r_lse, 4e-6, 2e-7, "logsumexp")


SHAPES = [(1, 1), (5, 3), (4, 33), (9, 128), (33, 1000), (3, 1023), (4, 4096), (2, 8193),
          (3, 16384), (2, 32768), (1, 152064), (2, 300000)]


@pytest.mark.parametrize("io", [("f32", "f32"), ("f32", "bf16"), ("bf16", "f32"), ("bf16", "bf16")])
@pytest.mark.parametrize("M,N", SHAPES)
def test_log_softmax(M, N, io):
    x = case(M, N, io[0], seed_of("log", M, N, io))
    y = osr.log_softmax_rows(x.cuda(), out_dtype=DT[io[1]])
    torch.cuda.synchronize()
    check_log(x, y)


@pytest.mark.parametrize("spec", ["rows:g=512", "cluster:g=256,cs=5", "staged:cs=3", "split:s=6,b=4"])
def test_log_softmax_every_tier(spec):
    x = case(37, 5000, "f32", seed_of("logtier", spec))
    with osr.forced_kernel(spec):
        y = osr.log_softmax_rows(x.cuda())
        torch.cuda.synchronize()
    check_log(x, y)


def test_log_softmax_misaligned_and_in_place():
    x = case(6, 1001, "f32", 3)
    buf = torch.empty(6 * 1001 + 1, device="cuda")
    xm = buf[1:].view(6, 1001)
    xm.copy_(x.cuda())
    osr.log_softmax_rows(xm, out=xm)
    torch.cuda.synchronize()
    check_log(x, xm)


def test_log_softmax_minus_inf():
    x = torch.tensor([[0.0, -float("inf"), 1.0, 2.0]], device="cuda")
    y = osr.log_softmax_rows(x).cpu()
    assert y[0, 1] == -float("inf")
    assert abs(float(torch.logsumexp(y[0, [0, 2, 3]].double(), 0))) < 1e-6


@pytest.mark.parametrize("dt", ["f32", "bf16"])
@pytest.mark.parametrize("M,N", [(1, 1), (7, 2), (100, 32), (33, 1000), (3, 1023), (64, 4096),
                                 (16, 2048), (9, 32768), (4, 152064), (1, 152064), (2, 300000),
                                 (300, 5000)])
def test_row_logsumexp(M, N, dt):
    x = case(M, N, dt, seed_of("lse", M, N, dt))
    lse, am = osr.row_logsumexp(x.cuda())
    torch.cuda.synchronize()
    check_lse(x, lse, am)


def test_row_logsumexp_only_one_output_and_misaligned():
    x = case(10, 3001, "bf16", 5)
    buf = torch.empty(10 * 3001 + 1, dtype=torch.bfloat16, device="cuda")
    xm = buf[1:].view(10, 3001)
    xm.copy_(x.cuda())
    lse, am = osr.row_logsumexp(xm, want_argmax=False)
    assert am is None
    _, am2 = osr.row_logsumexp(xm, want_lse=False)
    torch.cuda.synchronize()
    check_lse(x, lse, am2)


def test_row_logsumexp_ties_and_edges():
    x = torch.tensor([[1.0, 5.0, 5.0, 2.0, 5.0],
                      [7.0, 7.0, 7.0, 7.0, 7.0],
                      [-float("inf")] * 5,
                      [0.0, float("nan"), 3.0, 3.0, 1.0]], device="cuda")
    lse, am = osr.row_logsumexp(x)
    lse, am = lse.cpu(), am.cpu()
    assert am.tolist()[:3] == [1, 0, -1]
    assert am[3] == 2                                        # NaN is skipped by the maximum
    assert lse[2] == -float("inf") and torch.isnan(lse[3])
    assert abs(float(lse[1]) - (7.0 + np.log(5.0))) < 1e-6
    # ties placed far apart so they fall to different threads and CTAs
    for N in (4096, 152064):
        row = torch.zeros(3, N, device="cuda")
        row[:, 7] = 9.0
        row[:, N - 5] = 9.0
        _, am = osr.row_logsumexp(row)
        assert am.cpu().tolist() == [7, 7, 7]


@pytest.mark.parametrize("name", [n for n, w in workloads.WORKLOADS.items() if w.op == "logsumexp"])
def test_logsumexp_workloads_full_size(name):
    # every row of every log-sum-exp workload, in the launch the benchmark
    # times, checked a block of rows at a time
    w = workloads.WORKLOADS[name]
    x = workloads.make(w)["x"]
    lse, am = osr.row_logsumexp(x.cuda())
    torch.cuda.synchronize()
    lse, am = lse.cpu(), am.cpu()
    step = max(1, (1 << 24) // w.N)
    for r0 in range(0, w.M, step):
        check_lse(x[r0:r0 + step], lse[r0:r0 + step], am[r0:r0 + step])


@pytest.mark.parametrize("dt", ["bf16", "f32"])
@pytest.mark.parametrize("off", [0, 1, 3, 5])
@pytest.mark.parametrize("M,N", [(3, 50257), (40, 4097), (2000, 1001), (9, 152065), (70, 8200)])
def test_logsumexp_peeled_rows(M, N, off, dt):
    # rows that do not start on a 16-byte boundary (a base offset of `off`
    # elements, or a ragged length): each row's aligned body in vectors, its
    # head and tail one element a lane -- the cluster, CTA and group forms.
    # Maxima planted in the head, the tail, and tied across head and tail.
    x = case(M, N, dt, seed_of("lse-peel", M, N, off, dt)).float()
    top = 4000.0
    x[0, 0] = top
    x[1, N - 1] = top
    x[2, 1] = top
    x[2, N - 2] = top
    x = x.to(DT[dt])
    buf = torch.empty(M * N + off, dtype=x.dtype, device="cuda")
    xd = buf[off:].view(M, N)
    xd.copy_(x.cuda())
    ragged = off * x.element_size() % 16 != 0 or N % (16 // x.element_size()) != 0
    assert osr.plan_describe(osr.OP_LOGSUMEXP, M, N, dt, vec_ok=off == 0).endswith("peel" if ragged else "vec")
    lse, am = osr.row_logsumexp(xd)
    torch.cuda.synchronize()
    assert am.cpu().tolist()[:3] == [0, N - 1, 1]
    check_lse(x, lse, am)


@pytest.mark.parametrize("dt", ["bf16", "f32"])
@pytest.mark.parametrize("M", [8, 9, 54, 55, 68, 69, 127, 128, 512])
def test_logsumexp_plan_boundaries(M, dt):
    # the row counts where the planner changes tier on vocabulary rows:
    # staged -> 10 streaming CTAs (to 68 bf16 / 54 fp32 rows) -> a power of
    # two -> wide CTAs
    N = 152064
    x = case(M, N, dt, seed_of("lse-bound", M, dt), sigma=4.0)
    lse, am = osr.row_logsumexp(x.cuda())
    torch.cuda.synchronize()
    check_lse(x, lse, am)


@pytest.mark.parametrize("g", [1, 2, 4, 8, 16, 32, 64, 128, 256, 512, 1024])
@pytest.mark.parametrize("dt,misaligned", [("bf16", False), ("f32", False), ("bf16", True)])
def test_logsumexp_forced_group_widths(g, dt, misaligned):
    # a thread streams many tiles; rows whose maximum sits in the first tile
    # (so its first index is searched in a reloaded tile), in the last one,
    # tied across tiles, and a ragged tail
    M, N = 37, 5003 if misaligned else 5000
    x = case(M, N, dt, seed_of("lse-g", g, dt, misaligned)).float()
    top = 4000.0  # above every sample, shifted rows (+1000) included
    x[0, 3] = top
    x[1, N - 1] = top
    x[2, 5] = top
    x[2, N - 7] = top
    x[3, 1] = top
    x[3, 2] = top
    x = x.to(DT[dt])
    xd = x.cuda()
    if misaligned:
        buf = torch.empty(M * N + 1, dtype=x.dtype, device="cuda")
        xd = buf[1:].view(M, N)
        xd.copy_(x.cuda())
    with osr.forced_kernel(f"lse:g={g}"):
        assert osr.plan_describe(osr.OP_LOGSUMEXP, M, N, dt, vec_ok=not misaligned).startswith(f"lse-rows g={g} ")
        lse, am = osr.row_logsumexp(xd)
        torch.cuda.synchronize()
    assert am.cpu().tolist()[:4] == [3, N - 1, 5, 1]
    check_lse(x, lse, am)


def test_log_softmax_vocab_workload_full_size():
    w = workloads.WORKLOADS["log_softmax_vocab_bf16_f32_64x152064"]
    x = workloads.make(w)["x"]
    y = osr.log_softmax_rows(x.cuda(), out_dtype=torch.float32)
    torch.cuda.synchronize()
    check_log(x, y)


@pytest.mark.parametrize("dt", ["bf16", "f32"])
def test_row_logsumexp_staged_edges(dt):
    # few rows: pieces staged in shared memory; a -inf row, a NaN, ties split
    # over CTAs, and a row whose maximum sits in the last piece
    N = 131072
    x = torch.randn(4, N, generator=torch.Generator().manual_seed(17)) * 3
    x[0] = -float("inf")
    x[1, 40000] = float("nan")
    x[2, 9] = 50.0
    x[2, N - 3] = 50.0
    x[3, N - 1] = 60.0
    x = x.to(DT[dt])
    assert osr.plan_describe(osr.OP_LOGSUMEXP, 4, N, dt).startswith("lse-staged")
    lse, am = osr.row_logsumexp(x.cuda())
    lse, am = lse.cpu(), am.cpu()
    assert am.tolist()[0] == -1 and lse[0] == -float("inf")
    assert torch.isnan(lse[1]) and am[1] == int(torch.argmax(torch.nan_to_num(x[1].float(), nan=-1e30)))
    assert am.tolist()[2:] == [9, N - 1]
    check_lse(x[2:], lse[2:], am[2:])


@pytest.mark.parametrize("spec", ["lse:cs=2", "lse:cs=3", "lse:cs=10", "lse:cs=12", "lse:cs=16",
                                  "lse:cs=4,st=0", "lse:cs=10,st=0"])
def test_logsumexp_forced_cluster_sizes(spec):
    x = case(6, 152064, "bf16", seed_of("lse-cs", spec))
    with osr.forced_kernel(spec):
        lse, am = osr.row_logsumexp(x.cuda())
        torch.cuda.synchronize()
    check_lse(x, lse, am)
