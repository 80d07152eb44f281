"""Pins of the oracle against facts fixed outside of it (CPU only).

Each test checks the oracle against a closed form, an invariant, brute force,
or an independent library routine, chosen so that a plausible slip in the
oracle (dropped term, wrong sign, unbiased instead of biased variance, double
rounding, transposed operand) fails at least one of them.
"""
import math

import numpy as np
import pytest
import torch

from oracle.bf16 import round_bf16, bf16_bits_to_f64
from oracle.evaluator import evaluate, eval_op, round_to
from bytecode_vm_jit_gb300 import workloads as W

pytestmark = pytest.mark.filterwarnings("ignore::RuntimeWarning")


def f64_of(inputs, name):
    arr, dt = inputs[name]
    return bf16_bits_to_f64(arr) if dt == "bf16" else np.asarray(arr, np.float64)


# ---------------------------------------------------------------- bf16 ------
def test_bf16_matches_torch_on_float32_values():
    rng = np.random.default_rng(11)
    bits = rng.integers(0, 2**32, size=200_000, dtype=np.uint64).astype(np.uint32)
    f = bits.view(np.float32)
    f = f[np.isfinite(f)]
    specials = np.array([0.0, -0.0, 1.0, -1.0, np.inf, -np.inf, 3.3895314e38,
                         3.4e38, -3.4e38, 1e-45, 1.17549435e-38, 9.2e-41,
                         2.0**-133, 2.0**-134, 3 * 2.0**-134], dtype=np.float32)
    f = np.concatenate([f, specials])
    ours = round_bf16(f.astype(np.float64))
    ref = torch.from_numpy(f.copy()).to(torch.bfloat16).to(torch.float64).numpy()
    assert np.array_equal(ours, ref, equal_nan=True)


def test_bf16_ties_to_even_and_no_double_rounding():
    one = 1.0
    # midpoint between 1 and 1+2^-7 -> 1 (even); between 1+2^-7 and 1+2^-6 -> 1+2^-6
    assert round_bf16(one + 2**-8) == one
    assert round_bf16(one + 3 * 2**-8) == one + 2**-6
    # just above a midpoint: must round up although a float32 detour would tie
    assert round_bf16(one + 2**-8 + 2**-40) == one + 2**-7
    assert round_bf16(-(one + 2**-8 + 2**-40)) == -(one + 2**-7)
    # subnormal spacing 2^-133: 2^-134 ties to 0, 3*2^-134 ties up to 2^-132
    assert round_bf16(2.0**-134) == 0.0
    assert round_bf16(3 * 2.0**-134) == 2.0**-132
    # overflow at the midpoint to 2^128
    assert round_bf16(float.fromhex("0x1.ffp127")) == np.inf
    assert round_bf16(float.fromhex("0x1.fefffp127")) == float.fromhex("0x1.fep127")
    assert np.isnan(round_bf16(np.nan))


# ------------------------------------------------------- elementwise ops ----
SPECIAL = [
    ("sqrt", [4.0, -1.0, np.inf, 0.0, -0.0], [2.0, np.nan, np.inf, 0.0, -0.0]),
    ("log", [1.0, 0.0, -1.0, np.inf], [0.0, -np.inf, np.nan, np.inf]),
    ("exp", [0.0, -np.inf, np.inf, 1000.0], [1.0, 0.0, np.inf, np.inf]),
    ("round", [0.5, 1.5, 2.5, -0.5, -1.5, 2.4999998], [0.0, 2.0, 2.0, -0.0, -2.0, 2.0]),
    ("floor", [-0.5, 1.9999999, -2.0], [-1.0, 1.0, -2.0]),
    ("abs", [-3.0, -0.0, -np.inf], [3.0, 0.0, np.inf]),
    ("neg", [1.0, 0.0], [-1.0, -0.0]),
    ("isfinite", [1.0, np.inf, -np.inf, np.nan, 0.0], [1.0, 0.0, 0.0, 0.0, 1.0]),
    ("rsqrt", [4.0, 0.0, np.inf], [0.5, np.inf, 0.0]),
    ("recip", [2.0, 0.0, -0.0], [0.5, np.inf, -np.inf]),
    ("silu", [0.0, -1000.0], [0.0, -0.0]),
]


@pytest.mark.parametrize("op,xs,want", SPECIAL)
def test_unary_special_values(op, xs, want):
    dt = "u8" if op == "isfinite" else "f32"
    got = eval_op(op, [np.array(xs, np.float64)], dt)
    want = np.array(want, np.float64)
    assert np.array_equal(got, want, equal_nan=True), (op, got, want)
    ok = ~np.isnan(want)
    assert np.array_equal(np.signbit(got[ok]), np.signbit(want[ok]))


def test_pow_c99_cases():
    a = np.array([-8.0, -2.0, 0.0, np.nan, 2.0, -np.inf])
    b = np.array([1.0 / 3.0, 2.0, -1.0, 0.0, 0.5, 3.0])
    got = eval_op("pow", [a, b], "f32")
    want = np.array([np.nan, 4.0, np.inf, 1.0, math.sqrt(2.0), -np.inf])
    want = want.astype(np.float32).astype(np.float64)
    assert np.array_equal(got, want, equal_nan=True)


def test_max_min_propagate_nan_and_scalar_order():
    a = np.array([np.nan, 1.0, 2.0])
    b = np.array([1.0, np.nan, 3.0])
    assert np.array_equal(eval_op("max", [a, b], "f32"), [np.nan, np.nan, 3.0], equal_nan=True)
    assert np.array_equal(eval_op("min", [a, b], "f32"), [np.nan, np.nan, 2.0], equal_nan=True)
    x = np.array([1.0, 5.0])
    assert np.array_equal(eval_op("subs", [x], "f32", (3.0, 1)), [2.0, -2.0])
    assert np.array_equal(eval_op("subs", [x], "f32", (3.0, 0)), [-2.0, 2.0])
    assert np.array_equal(eval_op("divs", [x], "f32", (10.0, 1)), [10.0, 2.0])
    assert np.array_equal(eval_op("pows", [np.array([4.0])], "f32", (-0.5, 0)), [0.5])
    # the scalar attribute is a float32 value
    got = eval_op("adds", [np.array([0.0])], "f32", (0.1, 0))
    assert got[0] == float(np.float32(0.1))


def test_each_op_rounds_once_to_its_dtype():
    x = np.array([1.0])
    assert eval_op("adds", [x], "f32", (2.0**-30, 0))[0] == 1.0
    # an fp64 result above a bf16 midpoint rounds up directly
    v = np.array([1.0 + 2**-8 + 2**-40])
    assert eval_op("cast", [v], "bf16")[0] == 1.0 + 2**-7
    assert eval_op("cast", [v], "f32")[0] == float(np.float32(v[0]))


def test_reductions_closed_form():
    x = np.arange(1.0, 9.0).reshape(2, 4)
    assert np.array_equal(eval_op("reduce_sum", [x], "f32"), [[10.0], [26.0]])
    assert np.array_equal(eval_op("reduce_mean", [x], "f32"), [[2.5], [6.5]])
    assert np.array_equal(eval_op("reduce_max", [x], "f32"), [[4.0], [8.0]])
    assert np.array_equal(eval_op("reduce_sum_all", [x], "f32"), [36.0])
    y = np.array([[1.0, np.nan, 3.0]])
    assert np.isnan(eval_op("reduce_max", [y], "f32")[0, 0])
    # Gauss: sum 1..n = n(n+1)/2 exactly
    n = 4096
    g = np.arange(1.0, n + 1.0)[None, :]
    assert eval_op("reduce_sum", [g], "f32")[0, 0] == n * (n + 1) / 2


# ------------------------------------------------------------ sqrt_add ------
def test_sqrt_add_exact_squares():
    rng = np.random.default_rng(5)
    k = rng.integers(0, 2049, size=(64, 128)).astype(np.float64)
    b = rng.integers(0, 4097, size=(64, 128)).astype(np.float64)
    a = k * k - b                       # exact in float32 (|values| < 2^24)
    inputs = {"a": (a.astype(np.float32), "f32"), "b": (b.astype(np.float32), "f32")}
    env = evaluate(W.SQRT_ADD_OPS, inputs)
    assert np.array_equal(env["y"], k)
    z = {"a": (np.zeros((3, 5), np.float32), "f32"), "b": (np.zeros((3, 5), np.float32), "f32")}
    assert np.array_equal(evaluate(W.SQRT_ADD_OPS, z)["y"], np.zeros((3, 5)))


def test_sqrt_add_random_within_fp32_rounding():
    inp = W.sqrt_add_inputs((64, 256), seed=0)
    env = evaluate(W.SQRT_ADD_OPS, inp)
    a, b = f64_of(inp, "a"), f64_of(inp, "b")
    ref = np.sqrt(a + b)        # mathematically exact target; oracle rounds twice
    assert np.max(np.abs(env["y"] - ref) / np.maximum(1, np.abs(ref))) < 2e-7


# ----------------------------------------------------------- layernorm ------
def _ln(x, gamma, beta):
    inp = {"x": (x.astype(np.float32), "f32"), "gamma": (gamma.astype(np.float32), "f32"),
           "beta": (beta.astype(np.float32), "f32")}
    return evaluate(W.LAYERNORM_OPS, inp)["y"]


def test_layernorm_arithmetic_sequence_biased_variance():
    n = 8
    x = np.arange(1.0, n + 1.0)[None, :]
    y = _ln(x, np.ones(n), np.zeros(n))
    var = (n * n - 1) / 12.0          # biased variance of 1..n
    assert abs(np.mean(y)) < 1e-6
    assert abs(np.mean(y * y) - var / (var + W.LAYERNORM_EPS)) < 1e-6
    # symmetry: y is odd about the middle element
    assert np.allclose(y[0], -y[0, ::-1], atol=1e-6)


def test_layernorm_invariants_random_rows():
    rng = np.random.default_rng(9)
    x = rng.standard_normal((16, 4096)).astype(np.float32) * 3 + 7
    y = _ln(x, np.ones(4096), np.zeros(4096))
    xs = x.astype(np.float64)
    var = np.var(xs, axis=1)          # numpy biased variance
    assert np.all(np.abs(y.mean(axis=1)) < 1e-5)
    assert np.allclose((y * y).mean(axis=1), var / (var + W.LAYERNORM_EPS), rtol=1e-5, atol=0)


def test_layernorm_constant_rows_give_beta_and_affine():
    rng = np.random.default_rng(3)
    beta = rng.standard_normal(256)
    gamma = rng.standard_normal(256)
    x = np.full((3, 256), 2.5)
    y = _ln(x, gamma, beta)
    assert np.array_equal(y, np.broadcast_to(beta.astype(np.float32).astype(np.float64), y.shape))
    x = rng.standard_normal((4, 256))
    y0 = _ln(x, np.ones(256), np.zeros(256))
    y1 = _ln(x, np.full(256, 2.0), np.full(256, 3.0))
    assert np.allclose(y1, 2 * y0 + 3, rtol=0, atol=1e-6)


def test_layernorm_matches_torch_library():
    gamma, beta, _ = W.layernorm_params()
    inp = W.layernorm_inputs(0, 37)
    env = evaluate(W.LAYERNORM_OPS, inp)
    x = torch.from_numpy(f64_of(inp, "x"))
    ref = torch.nn.functional.layer_norm(x, (4096,), torch.from_numpy(gamma.astype(np.float64)),
                                         torch.from_numpy(beta.astype(np.float64)),
                                         eps=W.LAYERNORM_EPS).numpy()
    assert np.max(np.abs(env["y"] - ref) / np.maximum(1, np.abs(ref))) < 2e-6


# ---------------------------------------------------------- qwen stream -----
def test_rmsnorm_invariants():
    rng = np.random.default_rng(21)
    t, d = 8, 512
    xb = W.f32_to_bf16_bits(rng.standard_normal((t, d)).astype(np.float32))
    rb = W.f32_to_bf16_bits(rng.standard_normal((t, d)).astype(np.float32))
    ones = W.f32_to_bf16_bits(np.ones(d, np.float32))
    g = W.f32_to_bf16_bits(np.zeros((t, 16), np.float32))
    base = {"x": (xb, "bf16"), "r": (rb, "bf16"), "w": (ones, "bf16"), "g": (g, "bf16"), "u": (g, "bf16")}
    env = evaluate(W.QWEN_STEP_OPS, base)
    h = env["h"]
    m = np.mean(h * h, axis=1)
    n = env["n"]
    assert np.allclose(np.mean(n * n, axis=1), m / (m + W.RMS_EPS), rtol=2e-2)
    # scaling x and r by 4 (exact in bf16) leaves n unchanged up to the eps term
    s4 = {k: v for k, v in base.items()}
    s4["x"] = (W.f32_to_bf16_bits(bf16_bits_to_f64(xb).astype(np.float32) * 4), "bf16")
    s4["r"] = (W.f32_to_bf16_bits(bf16_bits_to_f64(rb).astype(np.float32) * 4), "bf16")
    env4 = evaluate(W.QWEN_STEP_OPS, s4)
    assert np.array_equal(env4["h"], 4 * h)
    assert np.max(np.abs(env4["n"] - n)) <= 2 ** -7 * np.max(np.abs(n))
    # torch's rms_norm on the bf16-rounded h
    ref = torch.nn.functional.rms_norm(torch.from_numpy(h), (d,), eps=W.RMS_EPS).numpy()
    assert np.max(np.abs(n - ref) / np.maximum(np.abs(ref), 1e-3)) < 1e-2


def test_silu_mul_special_values_and_library():
    g = np.array([[0.0, 30.0, -1000.0, 1.0, -2.0, 5.0, 0.5, -0.5]])
    u = np.array([[3.0, 1.0, 7.0, 1.0, 1.0, 2.0, -1.0, 4.0]])
    gb = W.f32_to_bf16_bits(g.astype(np.float32))
    ub = W.f32_to_bf16_bits(u.astype(np.float32))
    one = W.f32_to_bf16_bits(np.ones(8, np.float32))
    inp = {"x": (one[None, :], "bf16"), "r": (one[None, :], "bf16"), "w": (one, "bf16"),
           "g": (gb, "bf16"), "u": (ub, "bf16")}
    s = evaluate(W.QWEN_STEP_OPS, inp)["s"]
    assert s[0, 0] == 0.0 and s[0, 1] == 30.0 and s[0, 2] == 0.0
    ref = (torch.nn.functional.silu(torch.from_numpy(g)) * torch.from_numpy(u)).numpy()
    assert np.max(np.abs(s - ref) / np.maximum(np.abs(ref), 1e-6)) < 2 ** -8


# ---------------------------------------------------------- if-else-add -----
def test_if_else_takes_the_forced_branch():
    for i in range(4):
        inp = W.if_else_inputs(i, 64, d=256)
        env = evaluate(W.IF_ELSE_ADD_OPS, inp)
        x, z = f64_of(inp, "x"), f64_of(inp, "z")
        s = math.fsum(x.ravel())
        assert (s > 0) == (i % 2 == 0)
        assert (env["s"][0] > 0) == (s > 0)
        want = env["t"] if s > 0 else env["e"]
        assert np.array_equal(env["y"], want)
        # the branch value is the rounded sum / difference: exact in fp64
        exact = x + z if s > 0 else x - z
        assert np.array_equal(want, round_bf16(exact))


def test_select_nan_takes_else():
    a, b = np.ones(3), np.zeros(3)
    assert np.array_equal(eval_op("select_gt0", [np.array([np.nan]), a, b], "f32"), b)
    assert np.array_equal(eval_op("select_gt0", [np.array([0.0]), a, b], "f32"), b)


# ------------------------------------------------------------ matmul ------
def _brute(a, w):
    m, k = a.shape
    n = w.shape[1]
    out = np.zeros((m, n))
    for i in range(m):
        for j in range(n):
            out[i, j] = math.fsum(float(a[i, t]) * float(w[t, j]) for t in range(k))
    return out


@pytest.mark.parametrize("m,n,k", [(1, 7, 64), (7, 1, 129), (7, 7, 7), (2, 3, 128)])
def test_matmul_brute_force(m, n, k):
    rng = np.random.default_rng(m * 100 + n * 10 + k)
    wt = W.f32_to_bf16_bits(rng.standard_normal((n, k)).astype(np.float32))
    bias = W.f32_to_bf16_bits(rng.standard_normal(n).astype(np.float32))
    a = W.f32_to_bf16_bits(rng.standard_normal((m, k)).astype(np.float32))
    A, Wm, B = bf16_bits_to_f64(a), bf16_bits_to_f64(wt).T, bf16_bits_to_f64(bias)
    inp = {"A": (a, "bf16"), "W": (np.ascontiguousarray(wt.T), "bf16"), "bias": (bias, "bf16")}
    env = evaluate(W.MATMUL_ABS_OPS, inp)
    p = _brute(A, Wm)
    assert np.array_equal(env["p"], round_to(p, "f32"))
    assert np.array_equal(env["y"], round_bf16(round_to(np.abs(round_to(p, "f32") + B), "f32") * 0.5))


def test_matmul_identity_and_zero():
    rng = np.random.default_rng(1)
    k = 64
    a = W.f32_to_bf16_bits(rng.standard_normal((5, k)).astype(np.float32))
    bias = W.f32_to_bf16_bits(rng.standard_normal(k).astype(np.float32))
    eye = W.f32_to_bf16_bits(np.eye(k, dtype=np.float32))
    env = evaluate(W.MATMUL_ABS_OPS, {"A": (a, "bf16"), "W": (eye, "bf16"), "bias": (bias, "bf16")})
    A, B = bf16_bits_to_f64(a), bf16_bits_to_f64(bias)
    assert np.array_equal(env["y"], round_bf16(np.abs(A + B) * 0.5))
    zero = np.zeros_like(a)
    env = evaluate(W.MATMUL_ABS_OPS, {"A": (zero, "bf16"), "W": (eye, "bf16"), "bias": (bias, "bf16")})
    assert np.array_equal(env["y"], round_bf16(np.abs(B) * 0.5)[None, :].repeat(5, 0))


# ---------------------------------------------------------- generators ----
def test_generators_are_seeded_and_shaped():
    rows = W.layernorm_rows()
    assert len(rows) == 200 and all(1 <= r <= 32 * 2048 for r in rows)
    assert rows == W.layernorm_rows()
    t = W.if_else_rows()
    assert len(t) == 500 and min(t) >= 64 and max(t) <= 16384
    m = W.matmul_rows()
    assert len(m) == 100 and min(m) >= 1 and max(m) <= 8192
    q = W.qwen_tokens()
    assert len(q) == 2000 and min(q) >= 128 and max(q) <= 4096
    a = W.layernorm_inputs(3, 5)["x"][0]
    assert np.array_equal(a, W.layernorm_inputs(3, 5)["x"][0])
