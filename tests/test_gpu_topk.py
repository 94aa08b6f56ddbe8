"""Parity of the top-k sampling prologue (osr_row_topk) with the fp64 oracle.

values and indices: bit-exact (the selection is exact: a total order on the
inputs, nothing rounded decides it); probs: the binary32 softmax tolerance
(|err| <= 1e-6 + 1e-5 |ref|); lse: |err| <= 4e-6 + 2e-7 |ref|, as the
log-sum-exp kernel.  Shapes span one-CTA rows, clusters of 2..16 CTAs,
ragged pieces, the element-wise path, tie-heavy bf16 rows, masked (-inf)
rows, NaN and signed zeros, k = 1 (the argmax), k = N and k = 1024."""
import math
import os

import numpy as np
import pytest
import torch

import oracle
import online_softmax_row_gb300 as osr
import workloads
from parity import check_f32_abs, to_oracle_input

pytestmark = pytest.mark.gpu

DT = {"f32": torch.float32, "bf16": torch.bfloat16}


@pytest.fixture(scope="module", autouse=True)
def gpu():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    osr.library()
    torch.cuda.init()


def rows(M, N, dt, seed, ties=True, sigma=4.0):
    g = torch.Generator().manual_seed(seed)
    x = torch.randn(M, N, generator=g) * sigma
    if ties:  # a third of the entries on a coarse grid: many equal values
        sel = torch.rand(M, N, generator=g) < 0.33
        x[sel] = torch.round(x[sel] * 2) / 2
    return x.to(DT[dt])


def check(x_cpu, k, values, indices, probs, lse, what=""):
    xo = to_oracle_input(x_cpu).reshape(-1, x_cpu.shape[-1])
    r_v, r_i, r_p, r_l = oracle.topk(xo, k)
    gi = indices.cpu().numpy().reshape(r_i.shape)
    assert np.array_equal(gi, r_i), f"{what}: indices differ in {int((gi != r_i).sum())} places"
    gv = values.cpu().numpy().astype(np.float64).reshape(r_v.shape)
    same = (gv == r_v) | (np.isnan(gv) & np.isnan(r_v))
    assert same.all(), f"{what}: values differ"
    # the row's own numbers: -0 stays -0 (== does not tell it from +0)
    num = ~np.isnan(r_v)
    assert np.array_equal(np.signbit(gv[num]), np.signbit(r_v[num])), f"{what}: signs of zero differ"
    if probs is not None:
        check_f32_abs(probs.reshape(r_p.shape), r_p, 1e-6, 1e-5, f"{what} probs")
    if lse is not None:
        check_f32_abs(lse.reshape(r_l.shape), r_l, 4e-6, 2e-7, f"{what} lse")


def run_forced(spec, fn):
    with osr.forced_kernel(spec):
        out = fn()
        torch.cuda.synchronize()
        return out


@pytest.mark.parametrize("dt", ["f32", "bf16"])
@pytest.mark.parametrize("M,N,k", [(3, 17, 5), (5, 1, 1), (4, 1000, 50), (2, 4096, 4096 // 4),
                                   (7, 8200, 64), (64, 32000, 50), (2, 152064, 1024),
                                   (1, 152064, 50), (3, 300000, 100)])
def test_topk(M, N, k, dt):
    x = rows(M, N, dt, seed=M * 1000 + N + k)
    out = osr.row_topk(x.cuda(), k)
    torch.cuda.synchronize()
    check(x, k, *out, what=f"{M}x{N} k={k} {dt}")


@pytest.mark.parametrize("dt", ["f32", "bf16"])
@pytest.mark.parametrize("M,N,k", [(15, 152064, 50), (20, 152064, 50), (64, 152064, 50), (80, 152064, 50),
                                   (96, 152064, 50), (97, 152064, 50), (130, 152064, 50), (200, 32768, 50),
                                   (120, 65536, 64), (98, 5000, 8)])
def test_topk_many_rows(M, N, k, dt):
    # up to 96 rows, the planner's few-row sizes (15 rows: 8 CTAs a row; 20
    # rows: 6; 64 rows: 4 in bf16, 6 in fp32; 80 and 96 rows: 3 in bf16);
    # beyond, its rows-in-flight sizes (1, 3 or 6 CTAs a row here); every
    # row checked
    x = rows(M, N, dt, seed=M * 7 + N + k)
    out = osr.row_topk(x.cuda(), k)
    torch.cuda.synchronize()
    check(x, k, *out, what=f"{M}x{N} k={k} {dt}")


@pytest.mark.parametrize("cs", [1, 2, 3, 4, 8, 16])
@pytest.mark.parametrize("dt", ["f32", "bf16"])
def test_topk_forced_cluster_sizes(cs, dt):
    x = rows(4, 40000, dt, seed=cs)
    out = run_forced(f"topk:cs={cs}", lambda: osr.row_topk(x.cuda(), 300))
    check(x, 300, *out, what=f"cs={cs} {dt}")


@pytest.mark.parametrize("dt", ["f32", "bf16"])
def test_topk_element_path_and_offsets(dt):
    # odd row length and a buffer starting 2 elements into an allocation:
    # the element-wise loads, pieces not on vector boundaries
    x = rows(5, 5003, dt, seed=7)
    big = torch.empty(5 * 5003 + 2, dtype=x.dtype, device="cuda")
    xv = big[2:].view(5, 5003)
    xv.copy_(x.cuda())
    for spec in ("", "topk:cs=3"):
        fn = lambda: osr.row_topk(xv, 77)
        out = run_forced(spec, fn) if spec else fn()
        torch.cuda.synchronize()
        check(x, 77, *out, what=f"offset {spec or 'default'}")


def test_topk_k_one_is_argmax_and_k_n_is_softmax():
    x = rows(6, 3000, "bf16", seed=3)
    xc = x.cuda()
    v, i, p, l = osr.row_topk(xc, 1)
    _, am = osr.row_logsumexp(xc)
    torch.cuda.synchronize()
    assert torch.equal(i[:, 0], am)
    assert torch.all(p == 1.0)
    y = torch.randn(4, 97).cuda()
    v, i, p, l = osr.row_topk(y, 97)
    sm = osr.softmax_rows(y)
    torch.cuda.synchronize()
    assert torch.allclose(torch.gather(sm, 1, i), p, rtol=1e-5, atol=1e-6)


def test_topk_nan_signed_zero_and_masked_rows():
    x = torch.tensor([[1.0, 3.0, 3.0, -0.0, 0.0, float("nan"), 3.0, -float("inf")] * 4,
                      [-float("inf")] * 30 + [2.0, -1.0],
                      [0.0, -0.0] * 16], dtype=torch.float32)
    for dt in ("f32", "bf16"):
        xx = x.to(DT[dt])
        out = osr.row_topk(xx.cuda(), 12)
        torch.cuda.synchronize()
        check(xx, 12, *out, what=dt)


def test_topk_masked_vocabulary_rows():
    # top-k filtered rows: 64 finite entries, the rest -inf; k above 64 takes
    # -inf values (probability 0), lowest indices first
    x = workloads.softmax_inputs(8, 152064, "bf16", sigma=4.0, mask="keep:64", seed=5)["x"]
    for k in (50, 64, 100):
        out = osr.row_topk(x.cuda(), k)
        torch.cuda.synchronize()
        check(x, k, *out, what=f"masked k={k}")


def test_topk_outputs_optional_and_repeatable():
    x = rows(16, 50000, "bf16", seed=11).cuda()
    a = osr.row_topk(x, 40)
    b = osr.row_topk(x, 40, want_probs=False, want_lse=False)
    torch.cuda.synchronize()
    assert b[2] is None and b[3] is None
    assert torch.equal(a[0], b[0]) and torch.equal(a[1], b[1])
    c = osr.row_topk(x, 40)
    torch.cuda.synchronize()
    for u, v in zip(a, c):
        assert torch.equal(u, v)


def test_topk_workload_full_size():
    w = workloads.WORKLOADS["topk_vocab_bf16_64x152064_k50"]
    x = workloads.make(w)["x"]
    out = osr.row_topk(x.cuda(), w.k)
    torch.cuda.synchronize()
    check(x, w.k, *out, what=w.name)


@pytest.mark.parametrize("spec", ["", "topk:cs=2"])
def test_topk_constant_rows(spec):
    # every element equal: the k smallest columns.  With two CTAs of 1000
    # elements each the lists fit but all 2000 words tie (more than a
    # gathered list holds); with one CTA the list itself overflows.  Row 3
    # alternates -0 and +0 (equal numbers, each returned with its own sign).
    x = torch.full((4, 2000), 1.5, dtype=torch.bfloat16)
    x[1] = -2.0
    x[3] = torch.tensor([-0.0, 0.0] * 1000)
    fn = lambda: osr.row_topk(x.cuda(), 50)
    out = run_forced(spec, fn) if spec else fn()
    torch.cuda.synchronize()
    check(x, 50, *out, what=f"constant {spec or 'default'}")
    assert out[1].cpu().tolist() == [list(range(50))] * 4
    assert torch.signbit(out[0][3]).cpu().tolist() == [True, False] * 25


def test_topk_on_pinned_host_rows():
    # page-locked host rows go straight to the kernel (cp.async from host
    # memory over the host link): the same result as device rows
    import ctypes
    lib = osr.library()
    x = rows(4, 152064, "bf16", seed=21)
    hx = x.clone().pin_memory()
    hv = torch.empty(4, 50, dtype=torch.float32).pin_memory()
    hi = torch.empty(4, 50, dtype=torch.int64).pin_memory()
    hp = torch.empty(4, 50, dtype=torch.float32).pin_memory()
    hl = torch.empty(4, dtype=torch.float32).pin_memory()
    st = torch.cuda.current_stream().cuda_stream
    assert lib.osr_row_topk(hx.data_ptr(), hv.data_ptr(), hi.data_ptr(), hp.data_ptr(), hl.data_ptr(),
                            4, 152064, 50, 1, st) == 0
    torch.cuda.synchronize()
    dv, di, dp, dl = osr.row_topk(x.cuda(), 50)
    torch.cuda.synchronize()
    assert torch.equal(hi, di.cpu()) and torch.equal(hv, dv.cpu())
    assert torch.equal(hp, dp.cpu()) and torch.equal(hl, dl.cpu())
