"""The dispatcher over a sweep of shapes (host only, no GPU): every plan it
describes is one the kernels can run -- group widths, cluster sizes and
piece sizes inside the compiled and hardware limits, and enough threads or
CTAs to cover the row."""
import re

import pytest

import online_softmax_row_gb300 as osr

ROWS = [1, 2, 3, 8, 9, 16, 17, 31, 32, 33, 51, 52, 54, 55, 64, 68, 69, 96, 97, 127, 128, 129,
        255, 256, 512, 1000, 1024, 4096, 65536]
LENGTHS = [1, 2, 7, 8, 31, 32, 33, 100, 1000, 1023, 1024, 2048, 4095, 4096, 5000, 8192, 16384,
           32000, 32768, 50257, 65536, 131072, 152064, 262144, 300000]
EB = {"f32": 4, "bf16": 2}


def kv(plan, key):
    m = re.search(rf"\b{key}=(\d+)", plan)
    return int(m.group(1)) if m else None


@pytest.fixture(scope="module", autouse=True)
def lib():
    osr.library()


@pytest.mark.parametrize("dt", ["f32", "bf16"])
@pytest.mark.parametrize("vec", [True, False])
def test_logsumexp_plans_are_runnable(dt, vec):
    for M in ROWS:
        for N in LENGTHS:
            plan = osr.plan_describe(osr.OP_LOGSUMEXP, M, N, dt, vec_ok=vec)
            ragged = not vec or N % (16 // EB[dt])
            # rows not 16-byte aligned (or ragged) stream peeled bodies from 64 elements on
            assert plan.endswith("peel" if ragged and N >= 64 else "scalar" if ragged else "vec"), (M, N, plan)
            body = plan.endswith(("vec", "peel"))
            u = 16 // EB[dt] if body else 1
            g, cs = kv(plan, "g"), kv(plan, "cs")
            assert g and g & (g - 1) == 0 and 1 <= g <= 1024, plan
            assert cs and 1 <= cs <= 16, plan
            if plan.endswith("peel"):
                assert g >= u, (M, N, plan)  # a lane per edge element
            nunits = N // u
            if plan.startswith("lse-staged"):
                piece = kv(plan, "piece")
                assert plan.endswith("vec") and M <= 8 and cs > 1 and 128 + piece <= 200 << 10, (M, N, plan)
                assert cs * piece // 16 >= nunits, (M, N, plan)
            elif plan.startswith("lse-cluster"):
                assert g == 256 and cs > 1, plan
                assert cs <= -(-nunits // (256 * (32 // u))), (M, N, plan)  # a full tile each
            else:
                assert plan.startswith("lse-rows") and cs == 1, plan


@pytest.mark.parametrize("dt", ["f32", "bf16"])
def test_topk_plans_are_runnable(dt):
    for M in ROWS:
        for N in LENGTHS:
            if N * EB[dt] > 16 * (192 << 10):
                with pytest.raises(osr.OsrError):
                    osr.plan_describe(osr.OP_TOPK, M, N, dt)
                continue
            plan = osr.plan_describe(osr.OP_TOPK, M, N, dt)
            cs, piece = kv(plan, "cs"), kv(plan, "piece")
            assert 1 <= cs <= 16 and piece <= 192 << 10, (M, N, plan)
            assert cs * piece >= N * EB[dt], (M, N, plan)


@pytest.mark.parametrize("op", [osr.OP_RMSNORM, osr.OP_FUSED, osr.OP_SOFTMAX, osr.OP_LAYERNORM])
@pytest.mark.parametrize("dt", ["f32", "bf16"])
def test_row_op_plans_are_runnable(op, dt):
    for M in ROWS:
        for N in LENGTHS:
            for vec in (True, False):
                plan = osr.plan_describe(op, M, N, dt, vec_ok=vec)
                tier = plan.split()[0]
                assert tier in ("rows", "cluster", "staged", "split"), plan
                cs, g = kv(plan, "cs"), kv(plan, "g")
                if tier in ("cluster", "staged"):
                    assert 1 <= cs <= 16, (op, M, N, plan)
                if g is not None:
                    assert g & (g - 1) == 0 and 1 <= g <= 1024, (op, M, N, plan)
                if tier == "staged":
                    assert op == osr.OP_SOFTMAX and "vec" in plan, (op, M, N, plan)
                    assert kv(plan, "piece") <= 200 << 10, (op, M, N, plan)
