"""Strength of the oracle's pins: plant one plausible mistake at a time in a
copy of oracle.c (on the CPU), rebuild the copy, and check that at least one
pin of tests/test_oracle.py fails against it.  The oracle itself is not
modified; each mutant lives in a temporary directory."""
import os

import pytest

import oracle
import test_oracle as pins

# (name, text in oracle.c, replacement): each a slip someone could make
MUTANTS = [
    ("eps outside the square root",
     "double r = 1.0 / sqrt(ss / (double)H + eps);",
     "double r = 1.0 / (sqrt(ss / (double)H) + eps);"),
    ("mean over H-1",
     "double r = 1.0 / sqrt(ss / (double)H + eps);",
     "double r = 1.0 / sqrt(ss / (double)(H > 1 ? H - 1 : 1) + eps);"),
    ("gamma dropped",
     "y[j] = h[j] * r * elem(gamma, dt, j);",
     "y[j] = h[j] * r;"),
    ("denominator without the max shift",
     "for (int64_t j = 0; j < N; ++j) d += exp(elem(x, dt, i * N + j) - m);",
     "for (int64_t j = 0; j < N; ++j) d += exp(elem(x, dt, i * N + j));"),
    ("min instead of max",
     "        if (v > m) {\n            m = v;\n            at = j;",
     "        if (v < m || m == -INFINITY) {\n            m = v;\n            at = j;"),
    ("output index reversed",
     "row_max_sum(x, dt, i, N, &m, &d, 0);\n        for (int64_t j = 0; j < N; ++j) y[i * N + j] = exp(elem(x, dt, i * N + j) - m) / d;",
     "row_max_sum(x, dt, i, N, &m, &d, 0);\n        for (int64_t j = 0; j < N; ++j) y[i * N + j] = exp(elem(x, dt, i * N + (N - 1 - j)) - m) / d;"),
    ("online rescale with the wrong sign",
     "d = d * exp(m - mn) + exp(v - mn);",
     "d = d * exp(mn - m) + exp(v - mn);"),
    ("online start state (x1, 0)",
     "double m = elem(x, dt, i * N), d = 1.0;",
     "double m = elem(x, dt, i * N), d = 0.0;"),
    ("merge forgets to rescale the second side",
     "*d = d1 * exp(m1 - mm) + d2 * exp(m2 - mm);",
     "*d = d1 * exp(m1 - mm) + d2;"),
    ("merge keeps the smaller max",
     "double mm = m1 > m2 ? m1 : m2;",
     "double mm = m1 < m2 ? m1 : m2;"),
    ("bf16 rounded through binary32 first (double rounding)",
     "double r = nearbyint(v / q) * q;",
     "double r = nearbyint((double)(float)v / q) * q;"),
    ("bf16 ties away from zero",
     "double r = nearbyint(v / q) * q;",
     "double r = round(v / q) * q;"),
    ("fused normalises the unrounded sum",
     "h[j] = round_to(elem(x, dt, i * H + j) + elem(residual, dt, i * H + j), dt);",
     "h[j] = elem(x, dt, i * H + j) + elem(residual, dt, i * H + j);"),
    ("log-softmax drops log d",
     "y[i * N + j] = (elem(x, dt, i * N + j) - m) - ld;",
     "y[i * N + j] = (elem(x, dt, i * N + j) - m);"),
    ("logsumexp without the max",
     "if (lse) lse[i] = m + log(d);",
     "if (lse) lse[i] = log(d);"),
    ("argmax takes the last index on ties",
     "        if (v > m) {\n            m = v;\n            at = j;",
     "        if (v >= m) {\n            m = v;\n            at = j;"),
    ("layernorm variance about zero instead of the mean",
     "const double c = elem(x, dt, i * H + j) - mu;",
     "const double c = elem(x, dt, i * H + j);"),
    ("layernorm forgets beta",
     "* r * elem(gamma, dt, j) + elem(beta, dt, j);",
     "* r * elem(gamma, dt, j);"),
    ("welford uses the old mean in the M2 update",
     "m2 += delta * (v - mean);",
     "m2 += delta * delta;"),
    ("chan merge drops the between-group term",
     "*m2 = qa + qb + delta * delta * na * nb / nn;",
     "*m2 = qa + qb;"),
    ("top-k ties take the higher index first",
     "return a->i < b->i ? -1 : (a->i > b->i ? 1 : 0);",
     "return a->i > b->i ? -1 : (a->i < b->i ? 1 : 0);"),
    ("top-k sorted ascending",
     "if (!an && a->v != b->v) return a->v > b->v ? -1 : 1;",
     "if (!an && a->v != b->v) return a->v < b->v ? -1 : 1;"),
    ("top-k ranks NaN last",
     "if (an != bn) return an ? -1 : 1;",
     "if (an != bn) return an ? 1 : -1;"),
    ("top-k softmax normalised without the first value",
     "for (int64_t t = 0; t < k; ++t) z += exp(it[t].v - it[0].v);",
     "for (int64_t t = 1; t < k; ++t) z += exp(it[t].v - it[0].v);"),
    ("top-k softmax not shifted by the largest value",
     "if (probs) probs[i * k + t] = exp(it[t].v - it[0].v) / z;",
     "if (probs) probs[i * k + t] = exp(it[t].v) / z;"),
    ("chunk summary sums exp without its max",
     "for (int64_t j = c0; j < c1; ++j) cd += exp(elem(x, dt, i * N + j) - cm);",
     "for (int64_t j = c0; j < c1; ++j) cd += exp(elem(x, dt, i * N + j) - m);"),
]

PARAMS = {
    "test_softmax_invariants": [(31,), (257,)],
    "test_online_equals_three_pass": [(5,), (64,)],
    "test_chunk_summaries_merge_to_row_statistics": [(7,), (64,)],
    "test_softmax_matches_torch_fp64": [((3, 17),), ((8, 1000),)],
    "test_rmsnorm_matches_torch_rms_norm_fp64": [((5, 33), "f32"), ((5, 33), "bf16")],
    "test_logsumexp_constant_row_closed_form": [(7,)],
    "test_log_softmax_and_logsumexp_match_torch_fp64": [((3, 17),)],
    "test_layernorm_matches_torch_fp64": [((3, 33), "f32")],
    "test_topk_matches_numpy_lexsort": [(3, 17, 5, "f32"), (4, 1000, 50, "bf16")],
    "test_topk_probs_and_lse_match_torch_fp64": [(7,)],
}


def run_pins():
    """Names of the pins that fail against the currently loaded oracle."""
    failed = []
    for name in sorted(dir(pins)):
        if not name.startswith("test_"):
            continue
        fn = getattr(pins, name)
        for args in PARAMS.get(name, [()]):
            try:
                fn(*args)
            except Exception:  # an assertion, or NaN/inf tripping a check
                failed.append(name)
                break
    return failed


def test_pins_pass_on_the_real_oracle():
    assert run_pins() == []


@pytest.mark.parametrize("name,old,new", MUTANTS, ids=[m[0] for m in MUTANTS])
def test_each_planted_mistake_is_caught(name, old, new, tmp_path):
    src = open(oracle.SRC, encoding="utf-8").read()
    assert src.count(old) == 1, f"mutation site for '{name}' not found exactly once"
    lib = oracle.compile_variant(src.replace(old, new), str(tmp_path / "libmutant.so"))
    with oracle.use_library(lib):
        failed = run_pins()
    assert failed, f"no pin catches: {name}"
