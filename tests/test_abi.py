"""C-ABI checks that need no GPU: the library builds/loads, exports every
entry point the headers declare, validates arguments before touching a
device, and the length-based dispatcher picks the documented tier."""
import ctypes
import glob
import os
import re

import pytest

import online_softmax_row_gb300 as osr
from online_softmax_row_gb300 import build as osr_build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    osr_build.build()
    return osr.library()


def declared_symbols():
    names = set()
    for h in glob.glob(os.path.join(ROOT, "include", "*.h")):
        text = open(h, encoding="utf-8").read()
        text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
        names |= set(re.findall(r"\b(osr_[a-z0-9_]+)\s*\(", text))
    return sorted(names)


def test_headers_declare_the_three_operations():
    names = declared_symbols()
    for n in ("osr_rmsnorm_fwd", "osr_fused_add_rmsnorm", "osr_softmax_rows"):
        assert n in names


def test_library_exports_every_declared_symbol(lib):
    for n in declared_symbols():
        assert hasattr(lib, n), n


def test_status_strings_and_version(lib):
    for s in range(7):
        assert lib.osr_status_string(s)
    assert lib.osr_version() >= 100


# ------------------------------------------------------------ validation
# These calls return before any CUDA call: pointers are never dereferenced.

F32, BF16 = 0, 1
P = 0x10000  # fake, never dereferenced


def test_m_zero_is_noop(lib):
    assert lib.osr_softmax_rows(None, None, 0, 5, F32, F32, None) == 0
    assert lib.osr_rmsnorm_fwd(None, None, ctypes.c_float(1e-6), None, 0, 5, F32, None) == 0
    assert lib.osr_fused_add_rmsnorm(None, None, None, ctypes.c_float(1e-6), None, 0, 5, BF16, None) == 0


def test_invalid_sizes_and_dtypes(lib):
    assert lib.osr_softmax_rows(P, P * 4, 1, 0, F32, F32, None) == 1       # N == 0
    assert lib.osr_softmax_rows(P, P * 4, -1, 4, F32, F32, None) == 1      # M < 0
    assert lib.osr_softmax_rows(P, P * 4, 1, 4, 7, F32, None) == 1         # dtype
    assert lib.osr_softmax_rows(None, P, 1, 4, F32, F32, None) == 1        # NULL x
    assert lib.osr_rmsnorm_fwd(P, None, ctypes.c_float(0), P * 4, 1, 4, F32, None) == 1
    assert lib.osr_fused_add_rmsnorm(P, None, P * 2, ctypes.c_float(0), P * 4, 1, 4, F32, None) == 1
    # sizes whose byte counts would not fit int64: refused before anything else
    assert lib.osr_softmax_rows(P, P * 4, 2 ** 30, 2 ** 30, F32, F32, None) == 4
    assert lib.osr_rmsnorm_fwd(P, P, ctypes.c_float(0), P * 4, 2 ** 40, 2 ** 20, F32, None) == 4
    assert lib.osr_softmax_rows(P, P * 4, 1, 2 ** 41, F32, F32, None) == 4


def test_alias_rules(lib):
    # softmax: partial overlap forbidden; in place needs equal dtypes
    assert lib.osr_softmax_rows(P, P + 4, 4, 16, F32, F32, None) == 3
    assert lib.osr_softmax_rows(P, P, 4, 16, BF16, F32, None) == 3
    # rmsnorm: y overlapping gamma
    assert lib.osr_rmsnorm_fwd(P, P * 2 + 8, ctypes.c_float(0), P * 2, 4, 16, F32, None) == 3
    # fused: residual overlapping x / out
    assert lib.osr_fused_add_rmsnorm(P, P + 64, P * 8, ctypes.c_float(0), P * 16, 4, 16, F32, None) == 3
    assert lib.osr_fused_add_rmsnorm(P, P * 4, P * 8, ctypes.c_float(0), P * 4, 4, 16, F32, None) == 3
    # stats overlapping x
    assert lib.osr_softmax_rows_stats(P, P * 4, P, None, 4, 16, F32, F32, None) == 3


def test_host_pointers_rejected(lib):
    # plain host memory is not device memory: rejected before any launch
    buf = (ctypes.c_float * 64)()
    out = (ctypes.c_float * 64)()
    a, b = ctypes.addressof(buf), ctypes.addressof(out)
    assert lib.osr_softmax_rows(a, b, 4, 16, F32, F32, None) in (1, 5)


def test_bench_copy_validation(lib):
    assert lib.osr_bench_copy(P, P * 4, 0, None) == 0
    assert lib.osr_bench_copy(P, P * 4, 24, None) == 1       # not a multiple of 16
    assert lib.osr_bench_copy(P + 4, P * 4, 32, None) == 1   # misaligned
    assert lib.osr_bench_copy(P, P + 16, 64, None) == 3      # overlap


# ------------------------------------------------------------ dispatcher

@pytest.mark.parametrize("n,tier", [
    (1, "rows g=1"), (32, "rows g=2"), (128, "rows g=8"), (1024, "rows g=64"),
    (4096, "rows g=256"), (16384, "cluster cs=4 g=256"), (32768, "staged cs=12"),
    (152064, "staged cs=8"), (262144, "staged cs=14"), (1 << 20, "split"),
])
def test_dispatch_tiers_softmax_f32(lib, n, tier):
    assert osr.plan_describe(osr.OP_SOFTMAX, 64, n, "f32").startswith(tier)


@pytest.mark.parametrize("m,n,want", [
    # part of each piece in registers: the fewest pieces of at most 76 KiB
    (2048, 32768, "staged cs=2 g=256 piece=65536B r=8 vec"),
    (441, 152064, "staged cs=8 g=256 piece=76032B r=8 vec"),
    (128, 65536, "staged cs=4 g=256 piece=65536B r=8 vec"),
    (256, 98304, "staged cs=6 g=256 piece=65536B r=8 vec"),
    (2048, 40960, "staged cs=3 g=256 piece=54624B r=8 vec"),     # ragged: 3414 + 3414 + 3412 units
    (64, 152064, "staged cs=8 g=256 piece=76032B r=8 vec"),
    # fewer CTAs than SMs: spread over 12 CTAs, 16 for one or two rows
    (16, 152064, "staged cs=12 g=256 piece=50688B r=8 vec"),
    (8, 65536, "staged cs=12 g=256 piece=21856B r=8 vec"),
    (1, 32768, "staged cs=16 g=256 piece=8192B r=8 vec"),
    (3, 800000, "staged cs=16 g=256 piece=200000B r=8 vec"),    # largest pieces
])
def test_dispatch_staged_shapes(m, n, want):
    assert osr.plan_describe(osr.OP_SOFTMAX, m, n, "f32") == want


@pytest.mark.parametrize("m,n,io,want", [
    # bfloat16 rows stage whole pieces in shared memory: the fewest CTAs
    # reading and writing at most 80 KiB each, multiples of 4 above 8
    (441, 152064, ("bf16", "f32"), "staged cs=12 g=256 piece=25344B vec"),
    (512, 152064, ("bf16", "bf16"), "staged cs=8 g=256 piece=38016B vec"),
    (128, 262144, ("bf16", "bf16"), "staged cs=12 g=256 piece=43696B vec"),   # 13 -> 12
    (64, 152064, ("bf16", "f32"), "staged cs=12 g=256 piece=25344B vec"),     # few rows: 12 CTAs
    (2048, 32768, ("bf16", "f32"), "staged cs=3 g=256 piece=21856B vec"),
    (2048, 32768, ("bf16", "bf16"), "staged cs=2 g=256 piece=32768B vec"),
    (1024, 49152, ("bf16", "bf16"), "staged cs=3 g=256 piece=32768B vec"),
    (8192, 20480, ("bf16", "bf16"), "staged cs=1 g=256 piece=40960B vec"),
    (200, 400000, ("bf16", "f32"), "staged cs=16 g=256 piece=50000B vec"),    # as many as there are
    # fp32 -> bfloat16 holds part in registers like fp32 -> fp32
    (441, 152064, ("f32", "bf16"), "staged cs=8 g=256 piece=76032B r=8 vec"),
])
def test_dispatch_staged_shapes_by_dtype(m, n, io, want):
    assert osr.plan_describe(osr.OP_SOFTMAX, m, n, *io) == want


def test_dispatch_long_rows_without_staging():
    # norms and misaligned rows keep the register-cached cluster tier: up to
    # 16 CTAs of 256 threads, CTAs of 1024 threads beyond that
    assert osr.plan_describe(osr.OP_RMSNORM, 64, 32768, "f32") == "cluster cs=8 g=256 ept=16 vec"
    assert osr.plan_describe(osr.OP_RMSNORM, 8, 131072, "f32") == "cluster cs=8 g=1024 ept=16 vec"
    assert osr.plan_describe(osr.OP_SOFTMAX, 64, 32768, "f32", vec_ok=False) == "cluster cs=8 g=256 ept=16 scalar"
    # rows that would need a 1024-thread CTA go to four 256-thread CTAs
    assert osr.plan_describe(osr.OP_RMSNORM, 2048, 16384, "f32") == "cluster cs=4 g=256 ept=16 vec"
    assert osr.plan_describe(osr.OP_RMSNORM, 2048, 8192, "f32") == "rows g=512 ept=16 vec"


def test_dispatch_capacity_counts_cached_elements():
    # 16-byte bf16 rows: 32 elements a thread (softmax caches them as binary32,
    # the norms keep them packed); the split softmax kernels stay at 16
    assert osr.plan_describe(osr.OP_SOFTMAX, 64, 16384, "bf16", "f32") == "rows g=512 ept=32 vec"
    assert osr.plan_describe(osr.OP_SOFTMAX, 64, 16384, "f32") == "cluster cs=4 g=256 ept=16 vec"
    assert osr.plan_describe(osr.OP_SOFTMAX, 2048, 32768, "bf16", "f32") == "staged cs=3 g=256 piece=21856B vec"
    assert osr.plan_describe(osr.OP_SOFTMAX, 64, 1 << 22, "bf16", "f32").startswith("split")
    assert "ept=16" in osr.plan_describe(osr.OP_SOFTMAX, 64, 1 << 22, "bf16", "f32")
    assert osr.plan_describe(osr.OP_RMSNORM, 64, 16384, "bf16") == "rows g=512 ept=32 vec"
    assert osr.plan_describe(osr.OP_RMSNORM, 64, 32768, "bf16") == "cluster cs=4 g=256 ept=32 vec"
    assert osr.plan_describe(osr.OP_RMSNORM, 64, 65536, "bf16") == "cluster cs=8 g=256 ept=32 vec"
    assert osr.plan_describe(osr.OP_RMSNORM, 64, 32767, "bf16") == "cluster cs=8 g=256 ept=16 scalar"
    assert osr.plan_describe(osr.OP_SOFTMAX, 64, 152064, "bf16", "f32").startswith("staged cs=12")


def test_dispatch_scalar_path_when_misaligned():
    assert osr.plan_describe(osr.OP_SOFTMAX, 8, 1023, "f32").endswith("scalar")
    assert osr.plan_describe(osr.OP_SOFTMAX, 8, 1024, "f32", vec_ok=False).endswith("scalar")
    assert osr.plan_describe(osr.OP_SOFTMAX, 8, 1024, "f32").endswith("vec")


def test_dispatch_norms():
    assert osr.plan_describe(osr.OP_FUSED, 8192, 4096, "bf16") == "rows g=256 ept=16 vec"
    assert osr.plan_describe(osr.OP_LAYERNORM, 8192, 4096, "bf16") == "rows g=128 ept=32 vec"
    assert osr.plan_describe(osr.OP_RMSNORM, 64, 3584, "f32") == "rows g=256 ept=16 vec"
    with pytest.raises(osr.OsrError):
        osr.plan_describe(osr.OP_RMSNORM, 64, 3584, "f32", "bf16")


def test_split_shape_bounds():
    d = osr.plan_describe(osr.OP_SOFTMAX, 3, 10_000_000, "f32")
    s = int(re.search(r"s=(\d+)", d).group(1))
    b = int(re.search(r"b=(\d+)", d).group(1))
    assert 1 <= s <= 512 and 1 <= b <= 3


@pytest.fixture
def force(lib):
    """Set a forced plan (osr_test_force_kernel); cleared after the test."""
    def set_spec(spec):
        assert lib.osr_test_force_kernel(spec.encode() if spec else None) == 0
    yield set_spec
    lib.osr_test_force_kernel(None)


def test_force_kernel_setter(lib, force):
    assert osr.plan_describe(osr.OP_SOFTMAX, 10, 5000, "f32").startswith("rows g=")
    force("split:s=7,b=3")
    assert osr.plan_describe(osr.OP_SOFTMAX, 10, 5000, "f32").startswith("split s=7 b=3")
    force("")  # an empty spec forces nothing
    assert osr.plan_describe(osr.OP_SOFTMAX, 10, 5000, "f32").startswith("rows g=")
    assert lib.osr_test_force_kernel(b"x" * 64) == 1  # longer than 63 characters
    force(None)
    assert osr.plan_describe(osr.OP_SOFTMAX, 10, 5000, "f32").startswith("rows g=")


def test_forced_kernel(force):
    force("split:s=7,b=3")
    assert osr.plan_describe(osr.OP_SOFTMAX, 10, 5000, "f32").startswith("split s=7 b=3")
    force("cluster:g=256,cs=2")
    assert osr.plan_describe(osr.OP_SOFTMAX, 10, 5000, "f32").startswith("cluster cs=2 g=256")
    force("rows:g=512")
    assert osr.plan_describe(osr.OP_SOFTMAX, 10, 5000, "f32").startswith("rows g=512")
    # a forced shape that cannot hold the row is refused, not silently changed
    force("rows:g=64")
    with pytest.raises(osr.OsrError) as e:
        osr.plan_describe(osr.OP_SOFTMAX, 10, 5000, "f32")
    assert e.value.name == "OSR_ERR_UNSUPPORTED"
    force("cluster:g=256,cs=1")
    with pytest.raises(osr.OsrError):
        osr.plan_describe(osr.OP_SOFTMAX, 10, 5000, "f32")
    force("staged:cs=3")
    assert osr.plan_describe(osr.OP_SOFTMAX, 10, 5000, "f32").startswith("staged cs=3 g=256 piece=6672B")
    force("staged:cs=3,r=8")
    assert osr.plan_describe(osr.OP_SOFTMAX, 10, 5000, "f32") == "staged cs=3 g=256 piece=6672B r=8 vec"
    force("staged:cs=3,g=128,r=8")  # only the compiled shapes
    with pytest.raises(osr.OsrError):
        osr.plan_describe(osr.OP_SOFTMAX, 10, 5000, "f32")
    force("staged:cs=3,r=5")
    with pytest.raises(osr.OsrError):
        osr.plan_describe(osr.OP_SOFTMAX, 10, 5000, "f32")
    for bad in ((osr.OP_RMSNORM, True), (osr.OP_SOFTMAX, False)):  # softmax, 16-byte rows only
        with pytest.raises(osr.OsrError):
            osr.plan_describe(bad[0], 10, 5000, "f32", vec_ok=bad[1])
    force("staged:cs=17")
    with pytest.raises(osr.OsrError):
        osr.plan_describe(osr.OP_SOFTMAX, 10, 5000, "f32")


def test_logsumexp_plans_and_validation(lib):
    # staged for up to 8 rows long enough for 12 CTAs of full tiles (bf16
    # pieces 25 KiB: 8 an SM; fp32 pieces 50 KiB: 4 an SM); 10 streaming
    # CTAs a row while the grid fits one wave (bf16 up to 68 rows, fp32 up
    # to 54), then a power of two, about 512 CTAs in all
    assert osr.plan_describe(osr.OP_LOGSUMEXP, 8, 152064, "bf16") == "lse-staged g=256 cs=12 piece=25344B vec"
    assert osr.plan_describe(osr.OP_LOGSUMEXP, 9, 152064, "bf16") == "lse-cluster g=256 cs=10 vec"
    assert osr.plan_describe(osr.OP_LOGSUMEXP, 68, 152064, "bf16") == "lse-cluster g=256 cs=10 vec"
    assert osr.plan_describe(osr.OP_LOGSUMEXP, 69, 152064, "bf16") == "lse-cluster g=256 cs=4 vec"
    assert osr.plan_describe(osr.OP_LOGSUMEXP, 64, 152064, "bf16") == "lse-cluster g=256 cs=10 vec"
    assert osr.plan_describe(osr.OP_LOGSUMEXP, 96, 152064, "bf16") == "lse-cluster g=256 cs=4 vec"
    assert osr.plan_describe(osr.OP_LOGSUMEXP, 4, 32768, "bf16") == "lse-cluster g=256 cs=4 vec"  # too short to stage
    assert osr.plan_describe(osr.OP_LOGSUMEXP, 32, 152064, "f32") == "lse-cluster g=256 cs=10 vec"
    assert osr.plan_describe(osr.OP_LOGSUMEXP, 64, 32768, "bf16") == "lse-cluster g=256 cs=4 vec"  # a full tile each
    # from 128 rows: one CTA of up to 1024 threads per row (about 16 MB of
    # tiles in flight over the grid, two tiles a thread at least)
    assert osr.plan_describe(osr.OP_LOGSUMEXP, 128, 152064, "bf16") == "lse-rows g=1024 cs=1 vec"
    assert osr.plan_describe(osr.OP_LOGSUMEXP, 256, 152064, "bf16") == "lse-rows g=1024 cs=1 vec"
    assert osr.plan_describe(osr.OP_LOGSUMEXP, 512, 152064, "bf16") == "lse-rows g=512 cs=1 vec"
    assert osr.plan_describe(osr.OP_LOGSUMEXP, 1024, 152064, "bf16") == "lse-rows g=256 cs=1 vec"
    assert osr.plan_describe(osr.OP_LOGSUMEXP, 256, 152064, "f32") == "lse-rows g=512 cs=1 vec"
    assert osr.plan_describe(osr.OP_LOGSUMEXP, 256, 32768, "bf16") == "lse-rows g=512 cs=1 vec"
    assert osr.plan_describe(osr.OP_LOGSUMEXP, 256, 16384, "bf16") == "lse-cluster g=256 cs=2 vec"  # too short to widen
    assert osr.plan_describe(osr.OP_LOGSUMEXP, 54, 152064, "f32") == "lse-cluster g=256 cs=10 vec"
    assert osr.plan_describe(osr.OP_LOGSUMEXP, 55, 152064, "f32") == "lse-cluster g=256 cs=8 vec"
    assert osr.plan_describe(osr.OP_LOGSUMEXP, 1, 152064, "bf16") == "lse-staged g=256 cs=16 piece=19008B vec"
    assert osr.plan_describe(osr.OP_LOGSUMEXP, 8, 152064, "f32") == "lse-staged g=256 cs=12 piece=50688B vec"
    assert osr.plan_describe(osr.OP_LOGSUMEXP, 8, 152064, "f32", vec_ok=False) == "lse-cluster g=256 cs=10 peel"
    assert osr.plan_describe(osr.OP_LOGSUMEXP, 1024, 50257, "bf16") == "lse-rows g=256 cs=1 peel"  # ragged rows
    assert osr.plan_describe(osr.OP_LOGSUMEXP, 8, 63, "bf16", vec_ok=False) == "lse-rows g=2 cs=1 scalar"
    assert osr.plan_describe(osr.OP_LOGSUMEXP, 2, 3000000, "f32") == "lse-cluster g=256 cs=10 vec"  # pieces too big
    assert osr.plan_describe(osr.OP_LOGSUMEXP, 8192, 32000, "bf16") == "lse-rows g=256 cs=1 vec"
    assert osr.plan_describe(osr.OP_LOGSUMEXP, 100000, 32, "f32") == "lse-rows g=1 cs=1 vec"
    assert osr.plan_describe(osr.OP_LOG_SOFTMAX, 64, 4096, "f32") == "rows g=256 ept=16 vec"
    # both outputs NULL, overlapping outputs, NULL input
    assert lib.osr_row_logsumexp(P, None, None, 4, 16, F32, None) == 1
    assert lib.osr_row_logsumexp(None, P * 8, None, 4, 16, F32, None) == 1
    assert lib.osr_row_logsumexp(P, P + 8, None, 4, 16, F32, None) == 3
    assert lib.osr_row_logsumexp(P, P * 8, P * 8 + 4, 4, 16, F32, None) == 3
    assert lib.osr_row_logsumexp(P, P * 8, None, 0, 16, F32, None) == 0
    assert lib.osr_log_softmax_rows(P, P + 4, 4, 16, F32, F32, None) == 3


def test_layernorm_plans_and_validation(lib):
    assert osr.plan_describe(osr.OP_LAYERNORM, 256, 5120, "f32") == "rows g=512 ept=16 vec"
    assert osr.plan_describe(osr.OP_LAYERNORM, 4, 40000, "f32") == "cluster cs=10 g=256 ept=16 vec"
    assert osr.plan_describe(osr.OP_LAYERNORM, 2, 10 ** 6, "f32").startswith("split")
    f = ctypes.c_float(1e-5)
    assert lib.osr_layernorm_fwd(P, P * 8, None, f, P * 16, 4, 16, F32, None) == 1   # NULL beta
    assert lib.osr_layernorm_fwd(P, P * 8, P * 16 + 8, f, P * 16, 4, 16, F32, None) == 3  # y over beta
    assert lib.osr_layernorm_fwd(P, P * 8, P * 12, f, P + 4, 4, 16, F32, None) == 3      # y over x
    assert lib.osr_layernorm_fwd(None, None, None, f, None, 0, 16, F32, None) == 0


def test_topk_plans_and_validation(lib, force):
    D = osr.plan_describe
    assert D(osr.OP_TOPK, 64, 152064, "bf16") == "topk cs=4 piece=76032B vec"
    assert D(osr.OP_TOPK, 1, 152064, "bf16") == "topk cs=8 piece=38016B vec"    # few rows: 8 CTAs
    assert D(osr.OP_TOPK, 15, 152064, "bf16") == "topk cs=8 piece=38016B vec"   # one CTA an SM
    assert D(osr.OP_TOPK, 16, 152064, "f32") == "topk cs=6 piece=101376B vec"   # then 6 a row
    assert D(osr.OP_TOPK, 22, 152064, "bf16") == "topk cs=6 piece=50688B vec"
    assert D(osr.OP_TOPK, 23, 152064, "bf16") == "topk cs=4 piece=76032B vec"
    # the thresholds follow the SM count: half the SMs, half the rows
    assert [D(osr.OP_TOPK, m, 152064, "bf16", sm_count=76).split()[1] for m in (7, 8, 11, 12, 38, 39)] == \
        ["cs=8", "cs=6", "cs=6", "cs=4", "cs=4", "cs=3"]
    # many rows: the cluster size that keeps the most rows in flight per SM
    assert D(osr.OP_TOPK, 256, 152064, "bf16") == "topk cs=3 piece=101376B vec"
    assert D(osr.OP_TOPK, 256, 152064, "f32") == "topk cs=6 piece=101376B vec"
    assert D(osr.OP_TOPK, 2048, 32768, "bf16") == "topk cs=1 piece=65536B vec"
    assert D(osr.OP_TOPK, 2048, 65536, "bf16") == "topk cs=3 piece=43696B vec"
    assert D(osr.OP_TOPK, 2048, 262144, "bf16") == "topk cs=6 piece=87392B vec"
    # few rows: 4 CTAs a row while the grid stays one wave (two CTAs an SM
    # at 76 KiB pieces: 76 rows), then fewer; with no size fitting one wave,
    # the fewest CTAs per resident slot
    assert D(osr.OP_TOPK, 76, 152064, "bf16") == "topk cs=4 piece=76032B vec"
    assert D(osr.OP_TOPK, 77, 152064, "bf16") == "topk cs=3 piece=101376B vec"
    assert D(osr.OP_TOPK, 96, 152064, "bf16") == "topk cs=3 piece=101376B vec"
    assert D(osr.OP_TOPK, 32, 152064, "f32") == "topk cs=4 piece=152064B vec"
    assert D(osr.OP_TOPK, 64, 152064, "f32") == "topk cs=6 piece=101376B vec"
    assert D(osr.OP_TOPK, 8, 1000, "bf16") == "topk cs=1 piece=2000B vec"       # short rows: one CTA
    assert D(osr.OP_TOPK, 3, 33, "bf16", vec_ok=False) == "topk cs=1 piece=66B scalar"
    assert D(osr.OP_TOPK, 1, 786432, "f32") == "topk cs=16 piece=196608B vec"   # largest row
    with pytest.raises(osr.OsrError):
        D(osr.OP_TOPK, 1, 786433, "f32")                                        # beyond 16 x 192 KiB
    force("topk:cs=8")
    assert D(osr.OP_TOPK, 64, 152064, "bf16") == "topk cs=8 piece=38016B vec"
    force("lse:cs=16,st=0")
    assert osr.plan_describe(osr.OP_LOGSUMEXP, 64, 152064, "bf16") == "lse-cluster g=256 cs=16 vec"
    force("lse:cs=16,st=1")
    assert osr.plan_describe(osr.OP_LOGSUMEXP, 64, 152064, "bf16") == "lse-staged g=256 cs=16 piece=19008B vec"
    force("lse:cs=16")  # the staged form where the planner stages
    assert osr.plan_describe(osr.OP_LOGSUMEXP, 8, 152064, "bf16") == "lse-staged g=256 cs=16 piece=19008B vec"
    force("lse:g=32")
    assert osr.plan_describe(osr.OP_LOGSUMEXP, 64, 4096, "bf16") == "lse-rows g=32 cs=1 vec"
    force(None)
    T = lib.osr_row_topk
    assert T(P, P * 8, P * 16, None, None, 0, 16, 4, F32, None) == 0            # M == 0
    assert T(P, P * 8, P * 16, None, None, 4, 16, 0, F32, None) == 1            # k < 1
    assert T(P, P * 8, P * 16, None, None, 4, 16, 17, F32, None) == 1           # k > N
    assert T(P, P * 8, P * 16, None, None, 4, 4096, 1025, F32, None) == 4       # k > 1024
    assert T(P, None, P * 16, None, None, 4, 16, 4, F32, None) == 1             # NULL values
    assert T(P, P * 8, None, None, None, 4, 16, 4, F32, None) == 1              # NULL indices
    assert T(P, P + 8, P * 16, None, None, 4, 16, 4, F32, None) == 3            # values over x
    assert T(P, P * 8, P * 8 + 8, None, None, 4, 16, 4, F32, None) == 3         # indices over values
    assert T(P, P * 8, P * 16, P * 16 + 8, None, 4, 16, 4, F32, None) == 3      # probs over indices
    assert T(P, P * 8, P * 16, P * 24, P * 24, 4, 16, 4, F32, None) == 3        # lse over probs
