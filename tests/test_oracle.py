"""Pins for the fp64 oracle: the pages' worked examples (tests/golden/),
closed forms, invariants and library cross-checks.  CPU only.

Each check is chosen so that a plausible slip in the oracle -- a dropped
term, eps outside the square root, a wrong divisor, a missing max shift, a
wrong sign in a rescale factor, double rounding -- fails at least one of them.
"""
import itertools
import math
import os
import random

import numpy as np
import pytest
import torch

import oracle

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def load_golden(name):
    out = {}
    with open(os.path.join(GOLDEN, name), encoding="utf-8") as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            k, v = line.split(":", 1)
            out[k.strip()] = v.strip()
    return out


def nums(s):
    return [float(t) for t in s.split()]


def expr(s):
    """Evaluate an expression printed on a page: numbers, + - * /, exp()."""
    return float(eval(s, {"__builtins__": {}}, {"exp": math.exp}))


def f32(v):
    return np.asarray(v, dtype=np.float32)


def bf16_bits(t: torch.Tensor) -> np.ndarray:
    return t.contiguous().view(torch.int16).numpy().view(np.uint16)


def bits_to_f64(bits: np.ndarray) -> np.ndarray:
    return (bits.astype(np.uint32) << 16).view(np.float32).astype(np.float64)


# --------------------------------------------------------------- worked examples

def test_golden_rmsnorm_x3_4():
    g = load_golden("rmsnorm_x3_4.txt")
    tol = float(g["tol"])
    y, r = oracle.rmsnorm(f32(nums(g["x"])), f32(nums(g["gamma"])), float(g["eps"]),
                          return_rstd=True)
    assert abs(r[0] - float(g["expect.r"])) <= tol
    np.testing.assert_allclose(y[0], nums(g["expect.y"]), rtol=0, atol=tol)
    assert abs(np.mean(y[0] ** 2) - float(g["expect.mean_square_y"])) <= 1e-15


def test_golden_softmax_1000_1001():
    g = load_golden("softmax_1000_1001.txt")
    tol = float(g["tol"])
    y, m, d = oracle.softmax(f32(nums(g["x"])), return_stats=True)
    assert m[0] == float(g["expect.m"])
    assert abs(d[0] - float(g["expect.d"])) <= tol
    np.testing.assert_allclose(y[0], nums(g["expect.y"]), rtol=0, atol=tol)


def test_golden_online_stream_1_3_2():
    g = load_golden("online_stream_1_3_2.txt")
    tol = float(g["tol"])
    x = f32(nums(g["x"]))
    _, m2, d2 = oracle.softmax_online(x[:2], return_stats=True)
    assert m2[0] == float(g["expect.prefix2_m"])
    assert abs(d2[0] - float(g["expect.prefix2_d"])) <= tol
    y, m, d = oracle.softmax_online(x, return_stats=True)
    assert m[0] == float(g["expect.m"])
    assert abs(d[0] - float(g["expect.d"])) <= tol
    np.testing.assert_allclose(y[0], nums(g["expect.y"]), rtol=0, atol=tol)
    # the three-pass definition reaches the same numbers
    y3, m3, d3 = oracle.softmax(x, return_stats=True)
    np.testing.assert_allclose(y3[0], nums(g["expect.y"]), rtol=0, atol=tol)
    assert abs(d3[0] - float(g["expect.d"])) <= tol


def test_golden_tile_merge():
    g = load_golden("tile_merge_13_2.txt")
    tol = float(g["tol"])
    _, ma, da = oracle.softmax(f32(nums(g["tile_a"])), return_stats=True)
    _, mb, db = oracle.softmax(f32(nums(g["tile_b"])), return_stats=True)
    assert ma[0] == float(g["expect.a_m"]) and abs(da[0] - expr(g["expect.a_d_expr"])) <= tol
    assert mb[0] == float(g["expect.b_m"]) and db[0] == float(g["expect.b_d"])
    m, d = oracle.md_merge((ma[0], da[0]), (mb[0], db[0]))
    assert m == float(g["expect.m"])
    assert abs(d - expr(g["expect.d_expr"])) <= tol
    # and in the other order (commutativity)
    m2, d2 = oracle.md_merge((mb[0], db[0]), (ma[0], da[0]))
    assert m2 == m and abs(d2 - d) <= tol


def test_golden_softmax_2_4_1():
    g = load_golden("softmax_2_4_1.txt")
    tol = float(g["tol"])
    x = f32(nums(g["x"]))
    y, m, d = oracle.softmax(x, return_stats=True)
    assert m[0] == float(g["expect.m"])
    assert abs(d[0] - float(g["expect.d"])) <= tol
    np.testing.assert_allclose(y[0], nums(g["expect.y"]), rtol=0, atol=tol)
    for k, key in ((1, "expect.prefix1_d"), (2, "expect.prefix2_d")):
        _, _, dk = oracle.softmax_online(x[:k], return_stats=True)
        assert abs(dk[0] - float(g[key])) <= tol


def test_golden_stream_1_2_5_3():
    g = load_golden("stream_1_2_5_3.txt")
    tol = float(g["tol"])
    for fn in (oracle.softmax, oracle.softmax_online):
        _, m, d = fn(f32(nums(g["x"])), return_stats=True)
        assert m[0] == float(g["expect.m"])
        assert abs(d[0] - float(g["expect.d"])) <= tol


def test_golden_merge_check_every_bracketing():
    g = load_golden("merge_check_1_2_5.txt")
    x = nums(g["x"])
    leaves = [(v, 1.0) for v in x]
    A, B, C = leaves
    trees = [
        oracle.md_merge(oracle.md_merge(A, B), C),
        oracle.md_merge(A, oracle.md_merge(B, C)),
        oracle.md_merge(oracle.md_merge(A, C), B),
        oracle.md_merge(C, oracle.md_merge(B, A)),
    ]
    for m, d in trees:
        assert m == float(g["expect.m"])
        assert abs(d - float(g["expect.d"])) <= float(g["tol.d"])
        assert abs(d * math.exp(m) - float(g["expect.T"])) <= float(g["tol.T"])


def test_golden_trace_1_3_2_5():
    g = load_golden("trace_1_3_2_5.txt")
    tol = float(g["tol"])
    x = f32(nums(g["x"]))
    trace = [oracle.softmax_online(x[:k], return_stats=True)[1][0] for k in range(1, len(x) + 1)]
    assert trace == nums(g["expect.m_trace"])
    _, m, d = oracle.softmax_online(x, return_stats=True)
    assert m[0] == float(g["expect.m"])
    assert abs(d[0] - expr(g["expect.d_expr"])) <= tol


# --------------------------------------------------------------- closed forms

def test_rmsnorm_eps_inside_sqrt_closed_form():
    # mean square 12.5, eps 12.5 -> r = 1/sqrt(25) = 0.2 exactly, y = (0.6, 0.8)
    y, r = oracle.rmsnorm(f32([3, 4]), f32([1, 1]), 12.5, return_rstd=True)
    assert r[0] == 0.2
    np.testing.assert_allclose(y[0], [0.6, 0.8], rtol=1e-15)


def test_rmsnorm_constant_row_closed_form():
    # x_j = c for all j: r = (c^2 + eps)^(-1/2); divisor is H (not H-1)
    H, c, eps = 37, 1e-3, 1e-6
    gamma = np.linspace(0.5, 1.5, H).astype(np.float32)
    x = np.full(H, c, dtype=np.float32)
    y = oracle.rmsnorm(x, gamma, eps)[0]
    cc = float(np.float32(c))
    want = cc / math.sqrt(cc * cc + eps) * gamma.astype(np.float64)
    np.testing.assert_allclose(y, want, rtol=1e-14)


def test_rmsnorm_gamma_scales_each_column():
    rng = np.random.default_rng(1)
    x = rng.standard_normal((3, 50)).astype(np.float32)
    g1 = np.ones(50, np.float32)
    g2 = rng.uniform(0.5, 1.5, 50).astype(np.float32)
    y1 = oracle.rmsnorm(x, g1, 1e-6)
    y2 = oracle.rmsnorm(x, g2, 1e-6)
    np.testing.assert_allclose(y2, y1 * g2.astype(np.float64), rtol=1e-15)


def test_softmax_two_element_closed_form():
    # softmax(a, b) = (1/(1+e^(b-a)), 1/(1+e^(a-b)))
    for a, b in ((0.0, 0.0), (-3.5, 2.25), (80.0, -80.0), (1e3, 1e3 + 1)):
        y = oracle.softmax(f32([a, b]))[0]
        aa, bb = float(np.float32(a)), float(np.float32(b))
        np.testing.assert_allclose(y, [1 / (1 + math.exp(bb - aa)), 1 / (1 + math.exp(aa - bb))],
                                   rtol=1e-15)


def test_softmax_uniform_row():
    for n in (1, 2, 7, 1000):
        y = oracle.softmax(np.full(n, 3.25, np.float32))[0]
        assert np.all(y == 1.0 / n)


# --------------------------------------------------------------- invariants

@pytest.mark.parametrize("n", [1, 2, 3, 31, 33, 257, 4099])
def test_softmax_invariants(n):
    rng = np.random.default_rng(n)
    x = (rng.standard_normal((4, n)) * 5).astype(np.float32)
    y = oracle.softmax(x)
    assert np.all(y > 0)
    np.testing.assert_allclose(y.sum(axis=1), 1.0, rtol=0, atol=1e-13)
    for i in range(x.shape[0]):
        o = np.argsort(x[i], kind="stable")
        assert np.all(np.diff(y[i][o]) >= 0)          # order preserved
        assert np.argmax(y[i]) == np.argmax(x[i])


def test_softmax_shift_invariance_is_exact():
    # x on a 2^-10 grid with |x| < 8, so x + 1024 is exact in binary32 and the
    # max-shifted differences are bit-identical
    rng = np.random.default_rng(7)
    x = (rng.integers(-8191, 8192, size=(5, 300)) / 1024.0).astype(np.float32)
    xs = (x.astype(np.float64) + 1024.0).astype(np.float32)
    assert np.all(xs.astype(np.float64) - 1024.0 == x.astype(np.float64))
    assert np.array_equal(oracle.softmax(x), oracle.softmax(xs))
    assert np.array_equal(oracle.softmax_online(x), oracle.softmax_online(xs))


def test_softmax_large_values_do_not_overflow():
    x = np.array([[1000.0, 999.0, 1001.0, 1002.5], [-1e30, 0.0, 80.0, 88.0]], np.float32)
    y = oracle.softmax(x)
    assert np.all(np.isfinite(y))
    np.testing.assert_allclose(y.sum(axis=1), 1.0, atol=1e-15)


def test_rmsnorm_unit_mean_square_and_scale_invariance():
    rng = np.random.default_rng(3)
    x = rng.standard_normal((6, 129)).astype(np.float32)
    g = np.ones(129, np.float32)
    y = oracle.rmsnorm(x, g, 0.0)
    np.testing.assert_allclose(np.mean(y ** 2, axis=1), 1.0, rtol=0, atol=1e-14)
    # eps = 0: scaling a row by a power of two changes nothing, bit for bit
    assert np.array_equal(oracle.rmsnorm(x * np.float32(8.0), g, 0.0), y)


@pytest.mark.parametrize("n", [1, 2, 5, 64, 999])
def test_online_equals_three_pass(n):
    rng = np.random.default_rng(100 + n)
    x = (rng.standard_normal((3, n)) * 4).astype(np.float32)
    y3, m3, d3 = oracle.softmax(x, return_stats=True)
    yo, mo, do = oracle.softmax_online(x, return_stats=True)
    assert np.array_equal(m3, mo)
    np.testing.assert_allclose(do, d3, rtol=1e-13)
    np.testing.assert_allclose(yo, y3, rtol=1e-13)


@pytest.mark.parametrize("chunk", [1, 3, 4, 7, 64, 1000])
def test_chunk_summaries_merge_to_row_statistics(chunk):
    rng = np.random.default_rng(chunk)
    x = (rng.standard_normal((4, 1000)) * 6).astype(np.float32)
    _, m, d = oracle.softmax(x, return_stats=True)
    mc, dc = oracle.softmax_chunked_stats(x, chunk)
    assert np.array_equal(mc, m)
    np.testing.assert_allclose(dc, d, rtol=1e-13)


def test_merge_random_trees_identity_and_commutativity():
    rnd = random.Random(11)
    vals = [rnd.gauss(0, 6) for _ in range(60)]
    x = f32(vals)
    _, m_ref, d_ref = oracle.softmax(x, return_stats=True)
    for _ in range(20):
        # random split into pieces, each summarised, then merged in a random tree
        cuts = sorted(rnd.sample(range(1, 60), rnd.randint(1, 10)))
        pieces = [x[a:b] for a, b in zip([0] + cuts, cuts + [60])]
        summ = [tuple(v[0] for v in oracle.softmax(p, return_stats=True)[1:]) for p in pieces]
        while len(summ) > 1:
            i = rnd.randrange(len(summ) - 1)
            a, b = summ[i], summ[i + 1]
            if rnd.random() < 0.5:
                a, b = b, a
            summ[i:i + 2] = [oracle.md_merge(a, b)]
        m, d = summ[0]
        assert m == m_ref[0]
        assert abs(d - d_ref[0]) <= 1e-13 * d_ref[0]
    # (-inf, 0) is the identity
    for s in ((2.5, 1.75), (-40.0, 3.0)):
        assert oracle.md_merge((-math.inf, 0.0), s) == s
        assert oracle.md_merge(s, (-math.inf, 0.0)) == s


def test_denominator_at_least_one():
    rng = np.random.default_rng(5)
    x = (rng.standard_normal((20, 77)) * 30).astype(np.float32)
    _, m, d = oracle.softmax(x, return_stats=True)
    assert np.all(d >= 1.0)
    assert np.array_equal(m, x.max(axis=1).astype(np.float64))


def test_softmax_minus_inf_entries():
    x = np.array([[0.0, -np.inf, 1.0], [-np.inf, -np.inf, -np.inf]], np.float32)
    y = oracle.softmax(x)
    assert y[0, 1] == 0.0 and abs(y[0].sum() - 1) < 1e-15
    assert np.all(np.isnan(y[1]))


# --------------------------------------------------------------- library cross-checks

@pytest.mark.parametrize("shape", [(1, 1), (3, 17), (8, 1000), (2, 4096)])
def test_softmax_matches_torch_fp64(shape):
    g = torch.Generator().manual_seed(sum(shape))
    x = torch.randn(*shape, generator=g) * 7
    y = oracle.softmax(x.numpy())
    ref = torch.softmax(x.double(), dim=-1).numpy()
    np.testing.assert_allclose(y, ref, rtol=1e-13, atol=1e-300)


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("shape", [(1, 2), (5, 33), (4, 3584)])
def test_rmsnorm_matches_torch_rms_norm_fp64(shape, dtype):
    gen = torch.Generator().manual_seed(shape[1])
    x = torch.randn(*shape, generator=gen)
    w = torch.rand(shape[1], generator=gen) + 0.5
    if dtype == "bf16":
        x, w = x.bfloat16(), w.bfloat16()
        xa, wa = bf16_bits(x), bf16_bits(w)
    else:
        xa, wa = x.numpy(), w.numpy()
    y = oracle.rmsnorm(xa, wa, 1e-6)
    ref = torch.nn.functional.rms_norm(x.double(), (shape[1],), weight=w.double(), eps=1e-6)
    np.testing.assert_allclose(y, ref.numpy(), rtol=1e-13)


def test_fused_add_rmsnorm_matches_library_pieces():
    gen = torch.Generator().manual_seed(0)
    x = torch.randn(6, 256, generator=gen).bfloat16()
    r = torch.randn(6, 256, generator=gen).bfloat16()
    w = (torch.rand(256, generator=gen) + 0.5).bfloat16()
    h, y = oracle.fused_add_rmsnorm(bf16_bits(x), bf16_bits(r), bf16_bits(w), 1e-6)
    # new residual: the sum rounded once to bf16; torch adds in fp32, which is
    # exact for these operands, then rounds to bf16
    h_t = (x.float() + r.float()).bfloat16()
    assert np.array_equal(oracle.round_to(h, "bf16"), bf16_bits(h_t))
    # output: RMSNorm of the rounded sum
    ref = torch.nn.functional.rms_norm(h_t.double(), (256,), weight=w.double(), eps=1e-6)
    np.testing.assert_allclose(y, ref.numpy(), rtol=1e-13)
    # fp32 storage: the new residual is the fp32-rounded sum
    xf, rf = x.float().numpy() * 1.1, r.float().numpy()
    h32, _ = oracle.fused_add_rmsnorm(xf, rf, w.float().numpy(), 1e-6)
    assert np.array_equal(h32, (xf + rf).astype(np.float64))


# --------------------------------------------------------------- rounding

def test_round_bf16_matches_torch_on_binary32_values():
    g = torch.Generator().manual_seed(9)
    v = torch.cat([torch.randn(100000, generator=g) * 10.0 ** k for k in range(-40, 39, 6)])
    v = torch.cat([v, torch.tensor([0.0, -0.0, 1e-45, -1e-45, 3.3e38, -3.39e38])])
    ours = oracle.round_to(v.double().numpy(), "bf16")
    assert np.array_equal(ours, bf16_bits(v.bfloat16()))


def test_round_bf16_ties_overflow_subnormals_single_rounding():
    rb = oracle.round_bf16_bits
    assert rb(1.0 + 2.0 ** -8) == 0x3F80                  # tie -> even (down)
    assert rb(1.0 + 3 * 2.0 ** -8) == 0x3F82              # tie -> even (up)
    assert rb(1.0 + 2.0 ** -8 + 2.0 ** -40) == 0x3F81     # above the tie: one rounding only
    assert rb(-(1.0 + 2.0 ** -8 + 2.0 ** -40)) == 0xBF81
    assert rb((2 - 2.0 ** -8) * 2.0 ** 127) == 0x7F80     # halfway to 2^128 -> inf
    assert rb((2 - 2.0 ** -7) * 2.0 ** 127) == 0x7F7F     # largest finite
    assert rb(2.0 ** -133) == 0x0001                      # smallest subnormal
    assert rb(2.0 ** -134) == 0x0000                      # tie -> even (zero)
    assert rb(1.5 * 2.0 ** -134) == 0x0001
    assert rb(float("nan")) & 0x7FFF > 0x7F80
    assert rb(float("-inf")) == 0xFF80


def test_round_f32_matches_numpy():
    rng = np.random.default_rng(4)
    v = rng.standard_normal(10000) * 10.0 ** rng.integers(-45, 38, 10000)
    assert np.array_equal(oracle.round_to(v, "f32"), v.astype(np.float32))


def test_threads_do_not_change_results():
    rng = np.random.default_rng(8)
    x = rng.standard_normal((64, 500)).astype(np.float32)
    oracle.set_threads(1)
    a = oracle.softmax(x)
    oracle.set_threads(4)
    b = oracle.softmax(x)
    oracle.set_threads(1)
    assert np.array_equal(a, b)


def test_bit_helpers_agree_with_torch():
    t = torch.tensor([1.0, -2.5, 3.140625], dtype=torch.bfloat16)
    assert np.array_equal(bits_to_f64(bf16_bits(t)), t.double().numpy())
    assert list(itertools.islice(bf16_bits(t), 1)) == [0x3F80]


# --------------------------------------------------------------- log-softmax, logsumexp, argmax

def test_golden_logsumexp_1000_1001():
    g = load_golden("logsumexp_1000_1001.txt")
    tol = float(g["tol"])
    x = f32(nums(g["x"]))
    lse, am = oracle.logsumexp_argmax(x)
    assert am[0] == int(g["expect.argmax"])
    assert abs(lse[0] - (1001 + math.log(float(g["printed.d"])))) <= tol
    ly = oracle.log_softmax(x)[0]
    np.testing.assert_allclose(ly, [math.log(v) for v in nums(g["printed.y"])], rtol=0, atol=tol)


@pytest.mark.parametrize("n", [1, 2, 7, 1000])
def test_logsumexp_constant_row_closed_form(n):
    # n equal entries c: lse = c + log n, every log-probability is -log n
    c = 3.25
    lse, am = oracle.logsumexp_argmax(np.full(n, c, np.float32))
    assert abs(lse[0] - (c + math.log(n))) <= 1e-15 * (c + math.log(n))
    assert am[0] == 0                                  # first index on ties
    assert np.all(oracle.log_softmax(np.full(n, c, np.float32))[0] == -math.log(n))


@pytest.mark.parametrize("shape", [(1, 1), (3, 17), (8, 1000), (2, 4096)])
def test_log_softmax_and_logsumexp_match_torch_fp64(shape):
    g = torch.Generator().manual_seed(sum(shape) + 1)
    x = torch.randn(*shape, generator=g) * 7
    np.testing.assert_allclose(oracle.log_softmax(x.numpy()),
                               torch.log_softmax(x.double(), -1).numpy(), rtol=1e-13, atol=1e-13)
    lse, am = oracle.logsumexp_argmax(x.numpy())
    np.testing.assert_allclose(lse, torch.logsumexp(x.double(), -1).numpy(), rtol=1e-15)
    assert np.array_equal(am, np.argmax(x.numpy(), axis=1))


def test_log_softmax_is_log_of_softmax_and_shift_invariant():
    rng = np.random.default_rng(21)
    x = (rng.integers(-8191, 8192, size=(4, 300)) / 1024.0).astype(np.float32)
    ly = oracle.log_softmax(x)
    np.testing.assert_allclose(np.exp(ly), oracle.softmax(x), rtol=1e-14)
    xs = (x.astype(np.float64) + 1024.0).astype(np.float32)
    assert np.array_equal(oracle.log_softmax(xs), ly)
    lse, _ = oracle.logsumexp_argmax(x)
    lse_s, _ = oracle.logsumexp_argmax(xs)
    np.testing.assert_allclose(lse_s - 1024.0, lse, rtol=0, atol=1e-12)
    _, m, d = oracle.softmax(x, return_stats=True)
    np.testing.assert_allclose(lse, m + np.log(d), rtol=1e-15)


def test_argmax_first_index_on_ties_and_minus_inf():
    x = np.array([[1.0, 5.0, 5.0, 2.0], [-np.inf, -np.inf, 0.0, 0.0], [7.0, 7.0, 7.0, 7.0]],
                 np.float32)
    _, am = oracle.logsumexp_argmax(x)
    assert list(am) == [1, 2, 0]
    ly = oracle.log_softmax(x)
    assert ly[1, 0] == -np.inf and abs(ly[1, 2] + math.log(2)) < 1e-15


# --------------------------------------------------------------- LayerNorm, Welford, Chan

def ln_inputs(M, H, lo, hi, seed):
    rng = np.random.default_rng(seed)
    x = rng.uniform(lo, hi, (M, H)).astype(np.float32)
    g = rng.uniform(0.5, 1.5, H).astype(np.float32)
    b = rng.standard_normal(H).astype(np.float32)
    return x, g, b


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("shape", [(1, 2), (3, 33), (4, 5120)])
def test_layernorm_matches_torch_fp64(shape, dtype):
    gen = torch.Generator().manual_seed(shape[1] + 3)
    x = torch.rand(*shape, generator=gen) * 2 + 100     # mean ~101, the pages' stress case
    w = torch.rand(shape[1], generator=gen) + 0.5
    b = torch.randn(shape[1], generator=gen)
    if dtype == "bf16":
        x, w, b = x.bfloat16(), w.bfloat16(), b.bfloat16()
        xa, wa, ba = bf16_bits(x), bf16_bits(w), bf16_bits(b)
    else:
        xa, wa, ba = x.numpy(), w.numpy(), b.numpy()
    y = oracle.layernorm(xa, wa, ba, 1e-5)
    ref = torch.nn.functional.layer_norm(x.double(), (shape[1],), w.double(), b.double(), 1e-5)
    np.testing.assert_allclose(y, ref.numpy(), rtol=1e-12, atol=1e-12)


def test_layernorm_closed_forms():
    # constant row: x - mu = 0, y = beta
    H = 9
    g = np.linspace(0.5, 1.5, H).astype(np.float32)
    b = np.linspace(-1, 1, H).astype(np.float32)
    y = oracle.layernorm(np.full(H, 101.25, np.float32), g, b, 1e-5)[0]
    assert np.array_equal(y, b.astype(np.float64))
    # two elements a, b: mu = (a+b)/2, var = ((a-b)/2)^2, y = -+s/sqrt(s^2+eps) gamma + beta
    a, c, eps = 3.0, 7.0, 0.25
    s_ = (c - a) / 2
    y, mu, r = oracle.layernorm(f32([a, c]), f32([1, 1]), f32([0, 0]), eps, return_stats=True)
    assert mu[0] == 5.0 and r[0] == 1 / math.sqrt(s_ * s_ + eps)
    np.testing.assert_allclose(y[0], [-s_ * r[0], s_ * r[0]], rtol=1e-15)


def test_layernorm_standardises_and_is_shift_invariant():
    x, _, _ = ln_inputs(5, 1000, 100.0, 102.0, 4)
    ones, zeros = np.ones(1000, np.float32), np.zeros(1000, np.float32)
    y = oracle.layernorm(x, ones, zeros, 0.0)
    np.testing.assert_allclose(y.mean(axis=1), 0.0, atol=1e-12)
    np.testing.assert_allclose((y ** 2).mean(axis=1), 1.0, rtol=1e-12)
    # on a 2^-10 grid, x - 64 is exact and the output does not move
    xg = (np.round(x * 1024) / 1024).astype(np.float32)
    y1 = oracle.layernorm(xg, ones, zeros, 1e-5)
    y2 = oracle.layernorm((xg.astype(np.float64) - 64.0).astype(np.float32), ones, zeros, 1e-5)
    np.testing.assert_allclose(y1, y2, rtol=1e-10, atol=1e-10)


def test_welford_and_chan_merge_equal_two_pass():
    x, g, b = ln_inputs(3, 777, 100.0, 102.0, 5)
    _, mu, r = oracle.layernorm(x, g, b, 0.0, return_stats=True)
    var = 1 / r ** 2
    n, wm, m2 = oracle.welford(x)
    assert np.all(n == 777)
    np.testing.assert_allclose(wm, mu, rtol=1e-14)
    np.testing.assert_allclose(m2 / n, var, rtol=1e-10)
    # random splits merged in random trees (Chan) give the same statistics
    rnd = random.Random(6)
    for _ in range(10):
        cuts = sorted(rnd.sample(range(1, 777), rnd.randint(1, 12)))
        parts = [oracle.welford(x[0:1, a:b_]) for a, b_ in zip([0] + cuts, cuts + [777])]
        st = [(p[0][0], p[1][0], p[2][0]) for p in parts]
        while len(st) > 1:
            i = rnd.randrange(len(st) - 1)
            st[i:i + 2] = [oracle.chan_merge(st[i], st[i + 1])]
        nn, mm, qq = st[0]
        assert nn == 777 and abs(mm - mu[0]) <= 1e-13 * mu[0]
        assert abs(qq / nn - var[0]) <= 1e-9 * var[0]


# --------------------------------------------------------------- top-k prologue

def test_golden_topk_full_row_is_the_softmax_of_2_4_1_sorted():
    # with k = N the top-k softmax is the row's softmax, listed largest first
    g = load_golden("softmax_2_4_1.txt")
    x = f32(nums(g["x"]))[None, :]
    vals, idx, probs, lse = oracle.topk(x, 3)
    assert idx.tolist() == [[1, 0, 2]]
    assert vals.tolist() == [[4.0, 2.0, 1.0]]
    y = nums(g["expect.y"])
    np.testing.assert_allclose(probs[0], [y[1], y[0], y[2]], atol=float(g["tol"]))
    np.testing.assert_allclose(lse[0], 4.0 + math.log(float(g["expect.d"])), atol=1e-4)


def lexsort_topk(x: np.ndarray, k: int):
    """Library order: numpy's stable lexsort on (value descending, index)."""
    order = np.lexsort((np.arange(x.shape[1])[None, :].repeat(x.shape[0], 0), -x), axis=1)
    return order[:, :k]


@pytest.mark.parametrize("dt", ["f32", "bf16"])
@pytest.mark.parametrize("M,N,k", [(3, 17, 5), (4, 1000, 50), (2, 4096, 1024), (5, 64, 64)])
def test_topk_matches_numpy_lexsort(M, N, k, dt):
    g = torch.Generator().manual_seed(M * 7919 + N + k)
    x = torch.randn(M, N, generator=g) * 4
    x[:, ::7] = torch.round(x[:, ::7])  # plenty of equal values
    if dt == "bf16":
        xb = x.to(torch.bfloat16)       # bf16 rounding adds more ties
        arr, xs = bf16_bits(xb), xb.float().numpy().astype(np.float64)
    else:
        arr, xs = x.numpy(), x.numpy().astype(np.float64)
    vals, idx, probs, lse = oracle.topk(arr, k)
    want = lexsort_topk(xs, k)
    assert np.array_equal(idx, want)
    assert np.array_equal(vals, np.take_along_axis(xs, want, axis=1))


def test_topk_matches_torch_topk_on_distinct_values():
    g = torch.Generator().manual_seed(5)
    x = torch.randperm(5000, generator=g).reshape(5, 1000).float() * 0.25 - 300
    vals, idx, _, _ = oracle.topk(x.numpy(), 37)
    tv, ti = torch.topk(x.double(), 37, dim=1, sorted=True)
    assert np.array_equal(idx, ti.numpy())
    assert np.array_equal(vals, tv.numpy())


def test_topk_ties_nan_and_signed_zero():
    x = f32([[1.0, 3.0, 3.0, -0.0, 0.0, np.nan, 3.0, -np.inf]])
    vals, idx, _, _ = oracle.topk(x, 8)
    assert idx.tolist() == [[5, 1, 2, 6, 0, 3, 4, 7]]  # NaN first, equal values by index
    assert math.isnan(vals[0, 0]) and vals[0, 1:].tolist()[:4] == [3.0, 3.0, 3.0, 1.0]
    # k = 1 is the argmax (first index of the maximum) of a NaN-free row
    y = f32([[0.5, 2.0, -1.0, 2.0, 2.0]])
    assert oracle.topk(y, 1)[1].tolist() == [[1]]
    assert oracle.logsumexp_argmax(y)[1].tolist() == [1]


@pytest.mark.parametrize("k", [1, 7, 200])
def test_topk_probs_and_lse_match_torch_fp64(k):
    g = torch.Generator().manual_seed(k)
    x = torch.randn(6, 777, generator=g) * 5
    x[2, 100:] = -math.inf  # a masked row: the mass sits on the first 100
    vals, idx, probs, lse = oracle.topk(x.numpy(), k)
    np.testing.assert_allclose(probs, torch.softmax(torch.from_numpy(vals), -1).numpy(),
                               rtol=1e-14, atol=1e-300)
    np.testing.assert_allclose(probs.sum(axis=1), 1.0, rtol=1e-14)
    np.testing.assert_allclose(lse, torch.logsumexp(x.double(), -1).numpy(), rtol=1e-15)
    assert np.all(vals[:, 1:] <= vals[:, :-1])
