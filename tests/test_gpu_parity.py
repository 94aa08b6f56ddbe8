"""Parity of the CUDA path (through the C ABI) with the fp64 oracle, element
by element, on seeded inputs: small shapes spanning several tiles and ragged
tails, every dispatcher tier (forced), misaligned and in-place buffers, the
degenerate rows, and every benchmark workload at full size in the launch
configuration the benchmark times: every element of every row, compared in
chunks of rows, with the oracle running on all host cores."""
import os

import numpy as np
import pytest
import torch

import oracle
import online_softmax_row_gb300 as osr
import workloads
from parity import (seed_of, bits16, check_bf16, check_f32, check_out, check_row_max_and_argmax,
                    to_oracle_input)

pytestmark = pytest.mark.gpu

EPS = 1e-6
DT = {"f32": torch.float32, "bf16": torch.bfloat16}

SHAPES = [(1, 1), (7, 1), (5, 2), (3, 3), (4, 31), (4, 33), (9, 128), (33, 1000), (3, 1023),
          (64, 3584), (4, 4096), (2, 4097), (2, 8193), (3, 16384), (2, 32768), (2, 50000),
          (1, 152064), (2, 300000)]


@pytest.fixture(scope="module", autouse=True)
def gpu():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    osr.library()  # must be built: fail loudly otherwise
    torch.cuda.init()



def run_forced(spec, fn):
    with osr.forced_kernel(spec):
        out = fn()
        torch.cuda.synchronize()
        return out


# ------------------------------------------------------------ RMSNorm

def rms_case(M, N, dt, seed=0, fused=False, sigma=1.0):
    inp = workloads.rmsnorm_inputs(M, N, dt, sigma=sigma, fused=fused, seed=seed)
    return inp


def check_rmsnorm(inp, y):
    ref = oracle.rmsnorm(to_oracle_input(inp["x"]), to_oracle_input(inp["gamma"]), EPS)
    check_out(y, ref.reshape(y.shape), "rmsnorm")


def check_fused(inp, out, res_new):
    h_ref, y_ref = oracle.fused_add_rmsnorm(to_oracle_input(inp["x"]), to_oracle_input(inp["residual"]),
                                            to_oracle_input(inp["gamma"]), EPS)
    if res_new.dtype == torch.float32:
        assert np.array_equal(res_new.cpu().numpy().astype(np.float64), h_ref.reshape(res_new.shape))
    else:
        check_bf16(res_new, h_ref.reshape(res_new.shape), "residual")
        exact = np.mean(bits16(res_new).reshape(-1) == oracle.round_to(h_ref, "bf16").reshape(-1))
        assert exact >= 0.9999
    check_out(out, y_ref.reshape(out.shape), "fused out")


@pytest.mark.parametrize("dt", ["f32", "bf16"])
@pytest.mark.parametrize("M,N", SHAPES)
def test_rmsnorm(M, N, dt):
    inp = rms_case(M, N, dt, seed_of("rms", M, N, dt))
    y = osr.rmsnorm_fwd(inp["x"].cuda(), inp["gamma"].cuda(), EPS)
    check_rmsnorm(inp, y)


@pytest.mark.parametrize("dt", ["f32", "bf16"])
@pytest.mark.parametrize("M,N", SHAPES)
def test_fused_add_rmsnorm(M, N, dt):
    inp = rms_case(M, N, dt, seed_of("fused", M, N, dt), fused=True)
    res = inp["residual"].cuda()
    out = osr.fused_add_rmsnorm(inp["x"].cuda(), res, inp["gamma"].cuda(), EPS)
    check_fused(inp, out, res)


# ------------------------------------------------------------ softmax

def sm_case(M, N, dt, seed, sigma=4.0):
    return workloads.softmax_inputs(M, N, dt, sigma=sigma, shift_rows=M // 3, seed=seed)


def check_softmax(inp, y, rmax=None, rsum=None):
    xo = to_oracle_input(inp["x"]).reshape(y.shape[0], -1)
    ref, m, d = oracle.softmax(xo, return_stats=True)
    check_out(y, ref.reshape(y.shape), "softmax")
    if rmax is not None:
        check_row_max_and_argmax(xo, y, rmax, m, "softmax")
        s = rsum.cpu().numpy().astype(np.float64)
        assert np.all(np.abs(s - d) <= 1e-5 * d), "row sum"


@pytest.mark.parametrize("io", [("f32", "f32"), ("f32", "bf16"), ("bf16", "f32"), ("bf16", "bf16")])
@pytest.mark.parametrize("M,N", SHAPES)
def test_softmax(M, N, io):
    inp = sm_case(M, N, io[0], seed_of("sm", M, N, io))
    y, rmax, rsum = osr.softmax_rows_stats(inp["x"].cuda(), out_dtype=DT[io[1]])
    check_softmax(inp, y, rmax, rsum)


# ------------------------------------------------------------ every tier, forced

FORCED = ["rows:g=512", "rows:g=1024", "cluster:g=256,cs=2", "cluster:g=256,cs=5",
          "cluster:g=1024,cs=1", "cluster:g=1024,cs=3", "split:s=1,b=64", "split:s=3,b=5",
          "split:s=7,b=37", "split:s=40,b=2"]


@pytest.mark.parametrize("spec", FORCED)
@pytest.mark.parametrize("dt", ["f32", "bf16"])
def test_forced_tiers(spec, dt):
    M, N = 37, 5000
    inp = sm_case(M, N, dt, seed_of("forced", spec, dt))
    y, rmax, rsum = run_forced(spec, lambda: osr.softmax_rows_stats(inp["x"].cuda(),
                                                                    out_dtype=torch.float32))
    check_softmax(inp, y, rmax, rsum)
    ri = rms_case(M, N, dt, seed_of("forced-rms", spec, dt))
    y = run_forced(spec, lambda: osr.rmsnorm_fwd(ri["x"].cuda(), ri["gamma"].cuda(), EPS))
    check_rmsnorm(ri, y)
    fi = rms_case(M, N, dt, seed_of("forced-fused", spec, dt), fused=True)
    res = fi["residual"].cuda()
    out = run_forced(spec, lambda: osr.fused_add_rmsnorm(fi["x"].cuda(), res, fi["gamma"].cuda(), EPS))
    check_fused(fi, out, res)


@pytest.mark.parametrize("spec", ["staged:cs=1", "staged:cs=2", "staged:cs=5", "staged:cs=16",
                                  "staged:cs=3", "staged:cs=8", "staged:cs=1,r=0", "staged:cs=3,r=0",
                                  "staged:cs=16,r=0"])
@pytest.mark.parametrize("io", [("f32", "f32"), ("bf16", "f32"), ("f32", "bf16"), ("bf16", "bf16")])
def test_forced_staged(spec, io):
    M, N = 37, 5000
    inp = sm_case(M, N, io[0], seed_of("staged", spec, io))
    y, rmax, rsum = run_forced(spec, lambda: osr.softmax_rows_stats(inp["x"].cuda(),
                                                                    out_dtype=DT[io[1]]))
    check_softmax(inp, y, rmax, rsum)


# part of each piece held in registers: 5000-element rows fit the registers
# whole (no bulk copy at all); 40008-element rows leave a staged remainder,
# ragged over 3 pieces
@pytest.mark.parametrize("spec", ["staged:cs=1,r=8", "staged:cs=3,r=8", "staged:cs=2,r=8",
                                  "staged:cs=1,r=0", "staged:cs=3,r=0"])
@pytest.mark.parametrize("N", [5000, 40008])
@pytest.mark.parametrize("io", [("f32", "f32"), ("bf16", "f32"), ("f32", "bf16"), ("bf16", "bf16")])
def test_forced_staged_registers(spec, N, io):
    M = 5
    inp = sm_case(M, N, io[0], seed_of("staged-r", spec, N, io))
    y, rmax, rsum = run_forced(spec, lambda: osr.softmax_rows_stats(inp["x"].cuda(),
                                                                    out_dtype=DT[io[1]]))
    check_softmax(inp, y, rmax, rsum)


@pytest.mark.parametrize("spec", ["cluster:g=1024,cs=16", "split:s=512,b=1", "staged:cs=16,r=0",
                                  "staged:cs=16,r=8"])
def test_forced_limits(spec):
    M, N = 3, 200000
    inp = sm_case(M, N, "f32", seed_of("limits", spec))
    y, rmax, rsum = run_forced(spec, lambda: osr.softmax_rows_stats(inp["x"].cuda()))
    check_softmax(inp, y, rmax, rsum)


# ------------------------------------------------------------ layouts

def misaligned(t: torch.Tensor) -> torch.Tensor:
    """Same values at an address 1 element past a 16-byte boundary."""
    buf = torch.empty(t.numel() + 1, dtype=t.dtype, device="cuda")
    v = buf[1:].view(t.shape)
    v.copy_(t)
    return v


@pytest.mark.parametrize("N", [64, 1000, 4096, 40000])
@pytest.mark.parametrize("dt", ["f32", "bf16"])
def test_misaligned_buffers(N, dt):
    M = 6
    inp = sm_case(M, N, dt, seed_of("mis", N, dt))
    x = misaligned(inp["x"].cuda())
    assert x.data_ptr() % 16 != 0
    y = misaligned(torch.zeros(M, N, dtype=torch.float32, device="cuda"))
    osr.softmax_rows(x, out=y)
    check_softmax(inp, y)
    ri = rms_case(M, N, dt, seed_of("mis-rms", N, dt), fused=True)
    xr, res, g = misaligned(ri["x"].cuda()), misaligned(ri["residual"].cuda()), misaligned(ri["gamma"].cuda())
    out = osr.fused_add_rmsnorm(xr, res, g, EPS)
    check_fused(ri, out, res)


@pytest.mark.parametrize("N", [33, 4096, 32768, 300000])
@pytest.mark.parametrize("dt", ["f32", "bf16"])
def test_in_place(N, dt):
    M = 5
    inp = sm_case(M, N, dt, seed_of("inplace", N, dt))
    x = inp["x"].cuda()
    y = osr.softmax_rows(x, out=x)
    assert y.data_ptr() == x.data_ptr()
    check_softmax(inp, y)
    ri = rms_case(M, N, dt, seed_of("inplace-rms", N, dt))
    xr = ri["x"].cuda()
    osr.rmsnorm_fwd(xr, ri["gamma"].cuda(), EPS, out=xr)
    check_rmsnorm(ri, xr)
    fi = rms_case(M, N, dt, seed_of("inplace-fused", N, dt), fused=True)
    xf, res = fi["x"].cuda(), fi["residual"].cuda()
    osr.fused_add_rmsnorm(xf, res, fi["gamma"].cuda(), EPS, out=xf)
    check_fused(fi, xf, res)


def test_leading_dims_and_non_default_stream():
    inp = workloads.softmax_inputs(6 * 7, 257, "f32", sigma=3.0, seed=3)
    x = inp["x"].cuda().view(6, 7, 257)
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        y = osr.softmax_rows(x)
    s.synchronize()
    check_softmax(inp, y.view(42, 257))


def test_output_guard_pads_untouched():
    # outputs placed between poisoned pads; any out-of-range store shows up
    pad = 4096
    for N, dt in ((1000, "f32"), (4097, "bf16"), (40000, "f32"), (300000, "bf16")):
        M = 3
        inp = sm_case(M, N, dt, seed_of("pads", N, dt))
        big = torch.full((pad + M * N + pad,), 0x7FC01234, dtype=torch.int32, device="cuda")
        y = big[pad:pad + M * N].view(torch.float32).view(M, N)
        osr.softmax_rows(inp["x"].cuda(), out=y)
        torch.cuda.synchronize()
        assert torch.all(big[:pad] == 0x7FC01234) and torch.all(big[pad + M * N:] == 0x7FC01234)
        check_softmax(inp, y)


# ------------------------------------------------------------ degenerate rows

def test_edge_semantics_minus_inf_nan():
    x = torch.tensor([[0.0, -float("inf"), 1.0, 2.0],
                      [-float("inf")] * 4,
                      [1.0, float("nan"), 2.0, 3.0],
                      [5.0, 5.0, 5.0, 5.0]], device="cuda")
    y, rmax, _ = osr.softmax_rows_stats(x)
    y = y.cpu()
    assert y[0, 1] == 0 and abs(float(y[0].sum()) - 1) < 1e-6
    assert torch.isnan(y[1]).all()
    assert torch.isnan(y[2]).all()
    assert torch.all(y[3] == 0.25)
    assert rmax.cpu()[0] == 2.0 and rmax.cpu()[3] == 5.0


def test_empty_and_single_element_rows():
    x = torch.empty(0, 17, device="cuda")
    assert osr.softmax_rows(x).shape == (0, 17)
    assert osr.rmsnorm_fwd(x, torch.ones(17, device="cuda")).shape == (0, 17)
    x = torch.randn(1000, 1, device="cuda") * 100
    assert torch.all(osr.softmax_rows(x) == 1.0)


def test_errors_are_reported_not_fatal():
    x = torch.randn(4, 16, device="cuda")
    # in place across dtypes: the bf16 output overlaps the f32 input's rows
    y16 = x.view(-1).view(torch.bfloat16)[:64].view(4, 16)
    with pytest.raises(osr.OsrError) as e:
        osr.softmax_rows(x, out=y16, out_dtype=torch.bfloat16)
    assert e.value.name == "OSR_ERR_ALIAS"
    buf = torch.randn(100, device="cuda")
    with pytest.raises(osr.OsrError) as e:
        osr.softmax_rows(buf[:64].view(4, 16), out=buf[8:72].view(4, 16))
    assert e.value.name == "OSR_ERR_ALIAS"
    # the context still works afterwards
    check_softmax({"x": x.cpu()}, osr.softmax_rows(x))


def test_repeat_runs_bit_identical():
    for N, dt, spec in ((152064, "bf16", None), (4096, "f32", None), (300000, "f32", None),
                        (5000, "f32", "split:s=9,b=4")):
        inp = sm_case(8, N, dt, seed_of("det", N, dt))
        x = inp["x"].cuda()
        f = (lambda: osr.softmax_rows(x, out_dtype=torch.float32))
        runs = [run_forced(spec, f) if spec else f() for _ in range(5)]
        for r in runs[1:]:
            assert torch.equal(r.view(torch.int32), runs[0].view(torch.int32))


# ------------------------------------------------------------ full-size workloads

CHUNK_ELEMS = 8 << 20  # rows compared per step: about 64 MB of binary64 reference


@pytest.fixture
def oracle_all_cores():
    old = oracle.get_threads()
    oracle.set_threads(os.cpu_count() or 1)
    yield
    oracle.set_threads(old)


def check_softmax_rows_in_chunks(x_cpu, y, rmax, rsum, what):
    """Every element and every row statistic of a large softmax, a chunk of
    rows at a time (the oracle's binary64 output stays within memory)."""
    M, N = y.shape
    step = max(1, CHUNK_ELEMS // N)
    for r0 in range(0, M, step):
        r1 = min(M, r0 + step)
        check_softmax({"x": x_cpu[r0:r1]}, y[r0:r1], rmax[r0:r1], rsum[r0:r1])


@pytest.mark.parametrize("name", [n for n, w in workloads.WORKLOADS.items()
                                  if w.op in ("softmax", "rmsnorm", "fused_add_rmsnorm")])
def test_workload_full_size(name, oracle_all_cores):
    w = workloads.WORKLOADS[name]
    inp = workloads.make(w)
    if w.op == "softmax":
        if w.shift_rows:
            assert int((inp["x"][:, 0] > 500).sum()) == w.shift_rows
        x = inp["x"].cuda()
        y, rmax, rsum = osr.softmax_rows_stats(x, out_dtype=DT[w.out_dtype])
        torch.cuda.synchronize()
        del x
        check_softmax_rows_in_chunks(inp["x"], y, rmax, rsum, name)
        del y
    elif w.op == "rmsnorm":
        y = osr.rmsnorm_fwd(inp["x"].cuda(), inp["gamma"].cuda(), w.eps)
        check_rmsnorm(inp, y)
    else:
        res = inp["residual"].cuda()
        out = osr.fused_add_rmsnorm(inp["x"].cuda(), res, inp["gamma"].cuda(), w.eps)
        check_fused(inp, out, res)
    torch.cuda.empty_cache()


def test_pinned_host_buffers_zero_copy_and_pageable_refused():
    # page-locked host buffers go straight to the kernels (read and written
    # over the host link): the results are bit-identical to device buffers
    import ctypes
    lib = osr.library()
    st = torch.cuda.current_stream().cuda_stream
    inp = rms_case(64, 4096, "bf16", seed_of("host", 1), fused=True)
    hx, hr, hg = (inp[k].clone().pin_memory() for k in ("x", "residual", "gamma"))
    hy = torch.empty_like(hx).pin_memory()
    assert lib.osr_fused_add_rmsnorm(hx.data_ptr(), hr.data_ptr(), hg.data_ptr(), ctypes.c_float(EPS),
                                     hy.data_ptr(), 64, 4096, 1, st) == 0
    torch.cuda.synchronize()
    dr = inp["residual"].cuda()
    dy = osr.fused_add_rmsnorm(inp["x"].cuda(), dr, inp["gamma"].cuda(), EPS)
    torch.cuda.synchronize()
    assert torch.equal(hr, dr.cpu()) and torch.equal(hy, dy.cpu())
    xs = sm_case(8, 152064, "bf16", seed_of("host", 2))["x"]
    hx2 = xs.clone().pin_memory()
    hy2 = torch.empty(8, 152064, dtype=torch.float32).pin_memory()
    assert lib.osr_softmax_rows(hx2.data_ptr(), hy2.data_ptr(), 8, 152064, 1, 0, st) == 0
    torch.cuda.synchronize()
    assert torch.equal(hy2, osr.softmax_rows(xs.cuda(), out_dtype=torch.float32).cpu())
    # pageable host memory is refused before any launch
    px, py = xs.clone(), torch.empty(8, 152064, dtype=torch.float32)
    assert lib.osr_softmax_rows(px.data_ptr(), py.data_ptr(), 8, 152064, 1, 0, st) == 1
