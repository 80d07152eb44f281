"""Parity of the CUDA interpreter (through the C ABI) with the oracle, on GB300.

Tolerances (written here, from the path's contract): fp32 element-wise
|err| <= 1e-5 * max(1, |ref|); fp32 LayerNorm/RMSNorm <= 1e-4 * max(1, |ref|); bf16
outputs |err| <= 2e-2 * max(|ref|, rms(ref)).  Integer and branch decisions are exact.
"""
import numpy as np
import pytest
import torch

import bytecode_vm_jit_gb300 as D
from bytecode_vm_jit_gb300 import workloads as W
from oracle.bf16 import bf16_bits_to_f64
from oracle.evaluator import evaluate

pytestmark = [pytest.mark.gpu, pytest.mark.filterwarnings("ignore::RuntimeWarning")]


@pytest.fixture(scope="module", autouse=True)
def built():
    from bytecode_vm_jit_gb300 import build as B
    B.build()
    torch.cuda.set_device(0)


def to_dev(inputs):
    out = {}
    for k, (a, dt) in inputs.items():
        if dt == "bf16":
            out[k] = W.bf16_bits_to_torch(a).cuda()
        else:
            out[k] = torch.from_numpy(np.ascontiguousarray(a)).cuda()
    return out


def host(t):
    if t.dtype == torch.bfloat16:
        return bf16_bits_to_f64(t.view(torch.int16).cpu().numpy().view(np.uint16))
    return t.cpu().numpy().astype(np.float64)


def check_f32(got, ref, tol):
    err = np.abs(got - ref) / np.maximum(1.0, np.abs(ref))
    nan_ok = np.isnan(got) & np.isnan(ref)
    inf_ok = np.isinf(ref) & (got == ref)
    bad = ~((err <= tol) | nan_ok | inf_ok)
    assert not bad.any(), "max err %g at %s (got %r ref %r)" % (
        np.nanmax(np.where(nan_ok | inf_ok, 0, err)), np.argwhere(bad)[0], got[bad][0], ref[bad][0])


def check_bf16(got, ref):
    rms = np.sqrt(np.mean(ref ** 2)) if ref.size else 0.0
    bad = np.abs(got - ref) > 2e-2 * np.maximum(np.abs(ref), rms)
    assert not bad.any(), "bf16 mismatch at %s: got %r ref %r" % (np.argwhere(bad)[0], got[bad][0], ref[bad][0])


def run(ops, inputs, outputs, **kw):
    out = D.run_ops(ops, to_dev(inputs), outputs, **kw)
    torch.cuda.synchronize()
    return {k: host(v) for k, v in out.items()}


# ------------------------------------------------------------ sqrt_add -------
@pytest.mark.parametrize("shape", [(4096, 1024), (333, 1024), (5, 7), (1, 1), (3, 5, 130), (1000,)])
def test_sqrt_add(shape):
    inp = W.sqrt_add_inputs(shape, seed=0)
    got = run(W.SQRT_ADD_OPS, inp, W.SQRT_ADD_OUT)["y"]
    check_f32(got, evaluate(W.SQRT_ADD_OPS, inp)["y"], 1e-5)


def test_sqrt_add_exact_squares():
    rng = np.random.default_rng(5)
    k = rng.integers(0, 2049, size=(300, 1024)).astype(np.float64)
    b = rng.integers(0, 4097, size=(300, 1024)).astype(np.float64)
    inp = {"a": ((k * k - b).astype(np.float32), "f32"), "b": (b.astype(np.float32), "f32")}
    got = run(W.SQRT_ADD_OPS, inp, W.SQRT_ADD_OUT)["y"]
    assert np.array_equal(got, k)


def test_strided_input_uses_direct_loads():
    rng = np.random.default_rng(1)
    a = rng.random((256, 384), dtype=np.float32)
    b = rng.random((384, 256), dtype=np.float32)
    ta = torch.from_numpy(a).cuda()
    tb = torch.from_numpy(b).cuda().t()           # non-contiguous view
    out = D.run_ops(W.SQRT_ADD_OPS, {"a": ta, "b": tb}, W.SQRT_ADD_OUT)["y"]
    ref = evaluate(W.SQRT_ADD_OPS, {"a": (a, "f32"), "b": (np.ascontiguousarray(b.T), "f32")})["y"]
    check_f32(host(out), ref, 1e-5)


# ----------------------------------------------------------- layernorm -------
@pytest.mark.parametrize("rows", [1, 2, 37, 153, 1000])
def test_layernorm(rows):
    inp = W.layernorm_inputs(rows, rows)
    got = run(W.LAYERNORM_OPS, inp, W.LAYERNORM_OUT)["y"]
    check_f32(got, evaluate(W.LAYERNORM_OPS, inp)["y"], 1e-4)


def test_layernorm_invariants_and_reproducibility():
    rng = np.random.default_rng(3)
    x = (rng.standard_normal((64, 4096)) * 3 + 5).astype(np.float32)
    x[7] = 2.5                                   # constant row -> beta
    inp = {"x": (x, "f32"), "gamma": (np.ones(4096, np.float32), "f32"),
           "beta": (np.zeros(4096, np.float32), "f32")}
    y1 = run(W.LAYERNORM_OPS, inp, W.LAYERNORM_OUT)["y"]
    y2 = run(W.LAYERNORM_OPS, inp, W.LAYERNORM_OUT)["y"]
    assert np.array_equal(y1, y2)                # fixed reduction order
    rows = np.delete(np.arange(64), 7)
    assert np.all(np.abs(y1[rows].mean(axis=1)) < 1e-5)
    var = x[rows].astype(np.float64).var(axis=1)
    assert np.allclose((y1[rows] ** 2).mean(axis=1), var / (var + 1e-5), rtol=1e-4, atol=0)
    assert np.array_equal(y1[7], np.zeros(4096))


def test_layernorm_full_size_sampled_rows():
    """R = 65536 (largest instance): sampled rows against the oracle."""
    gamma, beta, _ = W.layernorm_params()
    g = torch.Generator(device="cuda")
    g.manual_seed(11)
    x = torch.randn(65536, 4096, device="cuda", generator=g)
    out = D.run_ops(W.LAYERNORM_OPS, {"x": x, "gamma": torch.from_numpy(gamma).cuda(),
                                      "beta": torch.from_numpy(beta).cuda()}, W.LAYERNORM_OUT)["y"]
    idx = torch.tensor([0, 1, 151, 152, 4097, 32768, 65534, 65535], device="cuda")
    xs = x[idx].cpu().numpy()
    ref = evaluate(W.LAYERNORM_OPS, {"x": (xs, "f32"), "gamma": (gamma, "f32"), "beta": (beta, "f32")})["y"]
    check_f32(out[idx].cpu().numpy().astype(np.float64), ref, 1e-4)


# ----------------------------------------------------------- if-else-add -----
@pytest.mark.parametrize("i,t", [(0, 64), (1, 64), (2, 300), (3, 1001), (4, 65), (5, 2048)])
def test_if_else_device_branch(i, t):
    inp = W.if_else_inputs(i, t)
    got = run(W.IF_ELSE_ADD_OPS, inp, W.IF_ELSE_ADD_OUT)["y"]
    ref = evaluate(W.IF_ELSE_ADD_OPS, inp)
    x = bf16_bits_to_f64(inp["x"][0])
    s = np.sum(x)
    tau = 2.0 ** -16 * np.sum(np.abs(x))
    if abs(s) > tau:
        assert np.array_equal(got, ref["y"])     # the forced branch, bit-exact
    else:
        assert np.array_equal(got, ref["t"]) or np.array_equal(got, ref["e"])


def test_if_else_full_size_sampled_rows():
    """T = 16384 (largest instance): the device branch follows the oracle's predicate over
    all of x, and sampled rows of y equal the oracle's chosen branch, bit for bit."""
    inp = W.if_else_inputs(7, 16384)
    dev = to_dev(inp)
    y = D.run_ops(W.IF_ELSE_ADD_OPS, dev, W.IF_ELSE_ADD_OUT)["y"]
    torch.cuda.synchronize()
    s_ref = evaluate(W.IF_ELSE_PRED_OPS, {"x": inp["x"]})["s"][0]
    x = bf16_bits_to_f64(inp["x"][0])
    assert abs(s_ref) > 2.0 ** -16 * np.sum(np.abs(x))       # the forced sign decides
    rows = np.array([0, 1, 151, 152, 8191, 8192, 16382, 16383])
    sample = {"x": (inp["x"][0][rows], "bf16"), "z": (inp["z"][0][rows], "bf16")}
    branch = W.IF_ELSE_THEN_OPS if s_ref > 0 else W.IF_ELSE_ELSE_OPS
    ref = evaluate(branch, sample)["y"]
    assert np.array_equal(host(y[torch.from_numpy(rows).cuda()]), ref)


def test_if_else_host_sync_variant_matches():
    inp = W.if_else_inputs(6, 500)
    dev = to_dev(inp)
    s = D.run_ops(W.IF_ELSE_PRED_OPS, {"x": dev["x"]}, ["s"])["s"]
    sv = float(s.cpu()[0])
    ops = W.IF_ELSE_THEN_OPS if sv > 0 else W.IF_ELSE_ELSE_OPS
    y_host = host(D.run_ops(ops, dev, ["y"])["y"])
    y_dev = host(D.run_ops(W.IF_ELSE_ADD_OPS, dev, W.IF_ELSE_ADD_OUT)["y"])
    assert np.array_equal(y_host, y_dev)
    ref = evaluate(W.IF_ELSE_PRED_OPS, inp)["s"][0]
    assert abs(sv - ref) <= 1e-3 * np.sum(np.abs(bf16_bits_to_f64(inp["x"][0]))) * 2 ** -10


def test_grid_barrier_timeout_is_reported_not_hung():
    inp = W.if_else_inputs(0, 300)
    dev = to_dev(inp)
    ctx = D.Ctx(0)
    try:
        D.dvm_debug_set_barrier(ctx.h, 1, 200)      # next barrier: one CTA never arrives
        ctx.feed(W.IF_ELSE_ADD_OPS, dev, W.IF_ELSE_ADD_OUT)
        assert ctx.poll() == -100
        D.dvm_debug_set_barrier(ctx.h, 0, 0)
        ctx.reset()
        out = ctx.feed(W.IF_ELSE_ADD_OPS, dev, W.IF_ELSE_ADD_OUT)
        assert ctx.poll() == 0
        assert np.array_equal(host(out["y"]), evaluate(W.IF_ELSE_ADD_OPS, inp)["y"])
    finally:
        ctx.close()


# ----------------------------------------------------------- qwen stream -----
@pytest.mark.parametrize("t", [1, 128, 333])
def test_qwen_step(t):
    inp = W.qwen_inputs(t, t)
    got = run(W.QWEN_STEP_OPS, inp, W.QWEN_STEP_OUT)
    ref = evaluate(W.QWEN_STEP_OPS, inp)
    for k in W.QWEN_STEP_OUT:
        check_bf16(got[k], ref[k])


def test_qwen_step_full_size_sampled_rows():
    """T = 4096 (largest step): every op is row-wise, so sampled token rows of h, n and s
    are checked against the oracle run on those rows alone."""
    inp = W.qwen_inputs(4096, 4096)
    dev = to_dev(inp)
    out = D.run_ops(W.QWEN_STEP_OPS, dev, W.QWEN_STEP_OUT)
    torch.cuda.synchronize()
    rows = np.array([0, 1, 151, 152, 2047, 2048, 4094, 4095])
    sample = {k: ((a[rows] if a.ndim == 2 else a), dt) for k, (a, dt) in inp.items()}
    ref = evaluate(W.QWEN_STEP_OPS, sample)
    idx = torch.from_numpy(rows).cuda()
    for k in W.QWEN_STEP_OUT:
        check_bf16(host(out[k][idx]), ref[k])


# ------------------------------------------------------------ op level -------
SPECIAL = np.array([0.0, -0.0, 1.0, -1.0, 0.5, 1.5, 2.5, -0.5, -2.5, 3.7, -3.7, 1e-30, 1e30,
                    np.inf, -np.inf, np.nan, 100.0, -100.0, 88.0, -87.0], dtype=np.float32)


@pytest.mark.parametrize("op", ["sqrt", "abs", "log", "exp", "round", "floor", "neg", "rsqrt", "recip", "silu"])
def test_unary_special_values(op):
    x = np.tile(SPECIAL, (3, 7))[:, :128].astype(np.float32)
    x = np.pad(x, ((0, 0), (0, 128 - x.shape[1])), constant_values=1.0)
    ops = [(op, ["x"], "y", "f32", ())]
    inp = {"x": (x, "f32")}
    got = run(ops, inp, ["y"])["y"]
    check_f32(got, evaluate(ops, inp)["y"], 2e-6)


def test_isfinite_and_binary_specials():
    x = np.tile(SPECIAL, 8)[None, :].astype(np.float32)
    y = np.roll(x, 3, axis=1)
    ops = [("isfinite", ["x"], "f", "u8", ()), ("pow", ["x", "y"], "p", "f32", ()),
           ("max", ["x", "y"], "mx", "f32", ()), ("min", ["x", "y"], "mn", "f32", ()),
           ("div", ["x", "y"], "d", "f32", ())]
    inp = {"x": (x, "f32"), "y": (y, "f32")}
    got = run(ops, inp, ["f", "p", "mx", "mn", "d"])
    ref = evaluate(ops, inp)
    assert np.array_equal(got["f"], ref["f"])
    for k in ("p", "mx", "mn", "d"):
        check_f32(got[k], ref[k], 2e-6)


def test_softmax_like_chain_rank3_ragged():
    rng = np.random.default_rng(4)
    x = rng.standard_normal((3, 5, 300)).astype(np.float32)
    c = rng.standard_normal((3, 5, 1)).astype(np.float32)
    ops = [("reduce_max", ["x"], "m", "f32", ()), ("sub", ["x", "m"], "d", "f32", ()),
           ("exp", ["d"], "e", "f32", ()), ("reduce_sum", ["e"], "s", "f32", ()),
           ("div", ["e", "s"], "p", "f32", ()), ("mul", ["p", "c"], "q", "f32", ()),
           ("subs", ["q"], "o", "f32", (1.0, 1))]
    inp = {"x": (x, "f32"), "c": (c, "f32")}
    got = run(ops, inp, ["o", "s"])
    ref = evaluate(ops, inp)
    check_f32(got["o"], ref["o"], 1e-5)
    check_f32(got["s"], ref["s"], 1e-5)


@pytest.mark.parametrize("rows,dt,d", [(37, "f32", 4096), (64, "f32", 4096), (45, "bf16", 8192)])
def test_softmax_rows_full_tiles(rows, dt, d):
    """Row max and row sum over complete one-row tiles (the packed and compile-time paths
    of the reduction handlers), a ragged last tile, and rows whose values are all
    negative (the max starts from -inf, not from 0)."""
    rng = np.random.default_rng(rows + d)
    x = (rng.standard_normal((rows, d)) * 3.0).astype(np.float32)
    x[1] = -np.abs(x[1]) - 5.0
    x[rows - 1] = -np.abs(x[rows - 1]) - 50.0
    if dt == "bf16":
        xb = W.f32_to_bf16_bits(x)
        inp = {"x": (xb, "bf16")}
    else:
        inp = {"x": (x, "f32")}
    ops = [("reduce_max", ["x"], "m", "f32", ()), ("sub", ["x", "m"], "z", "f32", ()),
           ("exp", ["z"], "e", "f32", ()), ("reduce_sum", ["e"], "s", "f32", ()),
           ("div", ["e", "s"], "p", "f32", ())]
    got = run(ops, inp, ["p", "m", "s"])
    ref = evaluate(ops, inp)
    check_f32(got["m"], ref["m"], 1e-6)
    check_f32(got["s"], ref["s"], 1e-5)
    check_f32(got["p"], ref["p"], 1e-5)
    assert np.all(got["m"][1] < 0) and np.all(got["m"][rows - 1] < -40)
