"""Parity of the CUBE kernel (MatMul tile op on tcgen05 + element-wise epilogue)
with the oracle, through the C ABI, on GB300.

Tolerance (bf16 outputs, fp32 accumulation): per element
|y - ref| <= 2e-2 * max(|ref|, rms(ref)); fp32 outputs of an epilogue that
ends in fp32: |err| <= 1e-3 * max(1, |ref|) relative to the fp64 oracle (the
products are accumulated in fp32 over K = 4096 terms, so the fp32 element-wise
bound of 1e-5 does not apply to the matmul itself).  Identity and zero weights
give exact results.
"""
import struct

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


def host(t):
    if t.dtype == torch.bfloat16:
        return bf16_bits_to_f64(t.view(torch.int16).cpu().numpy().view(np.uint16))
    return t.cpu().numpy().astype(np.float64)


def dev_bf16(bits):
    return W.bf16_bits_to_torch(np.ascontiguousarray(bits)).cuda()


def padded_bf16(bits, cols_pad):
    """[r, c] bf16 bits on the device as a view of an [r, cols_pad] buffer (row
    stride a multiple of 8 elements, as the MatMul operands require)."""
    r, c = bits.shape
    buf = np.zeros((r, cols_pad), np.uint16)
    buf[:, :c] = bits
    return dev_bf16(buf)[:, :c]


def check_bf16(got, ref):
    rms = np.sqrt(np.mean(ref ** 2)) if ref.size else 0.0
    bad = np.abs(got - ref) > 2e-2 * np.maximum(np.abs(ref), rms)
    assert not bad.any(), "bf16 mismatch at %s: got %r ref %r (of %d)" % (
        np.argwhere(bad)[0], got[bad][0], ref[bad][0], int(bad.sum()))


def run_mm(a_dev, w_dev, bias_dev, ops=W.MATMUL_ABS_OPS, extra=None):
    inputs = {"A": a_dev, "W": w_dev, "bias": bias_dev}
    if extra:
        inputs.update(extra)
    outs = ["y"]
    ctx = D.Ctx(0)
    try:
        out = ctx.feed(ops, inputs, outs)
        st = ctx.poll()
        assert st == 0, "device status %d" % st
        kinds = [img[6] for img, _ in ctx.launch_log]
    finally:
        ctx.close()
    torch.cuda.synchronize()
    assert kinds == [2], "expected one CUBE launch, got kernel types %r" % kinds
    return host(out["y"])


def oracle_mm(a_bits, wt_bits, bias_bits, ops=W.MATMUL_ABS_OPS, extra=None):
    inputs = {"A": (a_bits, "bf16"), "W": (np.ascontiguousarray(wt_bits.T), "bf16"), "bias": (bias_bits, "bf16")}
    if extra:
        inputs.update(extra)
    return evaluate(ops, inputs)["y"]


# ------------------------------------------------- the workload's shapes --
@pytest.mark.parametrize("m", [1, 7, 100, 128, 129, 300])
def test_matmul_abs(m):
    wt, bias, _ = W.matmul_params()
    inp = W.matmul_inputs(0, m, small_params=(wt, bias))
    a = inp["A"][0]
    got = run_mm(dev_bf16(a), dev_bf16(wt).t(), dev_bf16(bias))
    check_bf16(got, oracle_mm(a, wt, bias))


def test_matmul_abs_largest_instance_sampled_rows():
    """M = 8192 (largest instance, 1024 tiles of 128 x 256): 96 sampled rows."""
    wt, bias, _ = W.matmul_params()
    g = torch.Generator(device="cuda")
    g.manual_seed(17)
    a = (torch.randn(8192, 4096, device="cuda", generator=g) * 0.02).to(torch.bfloat16)
    got = run_mm(a, dev_bf16(wt).t(), dev_bf16(bias))
    rows = np.random.default_rng(3).choice(8192, 96, replace=False)
    rows = np.concatenate([rows, [0, 127, 128, 8191]])
    a_bits = a.view(torch.int16).cpu().numpy().view(np.uint16)[rows]
    check_bf16(got[rows], oracle_mm(a_bits, wt, bias))


# --------------------------------------------------- brute force, tiny shapes --
@pytest.mark.parametrize("m,n,k", [(1, 1, 1), (7, 7, 7), (64, 64, 64), (128, 128, 128), (129, 129, 129),
                                   (1, 129, 64), (129, 7, 128), (7, 300, 129), (200, 48, 1000),
                                   (5, 600, 3000), (130, 520, 2048)])
def test_matmul_brute_force(m, n, k):
    rng = np.random.default_rng(m * 10007 + n * 101 + k)
    a = W.f32_to_bf16_bits(rng.standard_normal((m, k)).astype(np.float32))
    wt = W.f32_to_bf16_bits(rng.standard_normal((n, k)).astype(np.float32))
    bias = W.f32_to_bf16_bits(rng.standard_normal(n).astype(np.float32))
    kp = (k + 7) // 8 * 8
    got = run_mm(padded_bf16(a, kp), padded_bf16(wt, kp).t(), dev_bf16(bias))
    af, wf, bf = bf16_bits_to_f64(a), bf16_bits_to_f64(wt), bf16_bits_to_f64(bias)
    ref = np.empty((m, n))
    for i in range(m):                       # triple loop, vectorised over k only
        for j in range(n):
            ref[i, j] = abs(float(np.dot(af[i], wf[j])) + bf[j]) * 0.5
    from oracle.bf16 import round_bf16
    check_bf16(got, round_bf16(ref))


def test_k_split_repeated_launches_agree():
    """Few-row MatMuls run as K-split tiles whose per-tile arrival counters live in the
    context's workspace and return to zero after every launch: the same instance run
    three times in one context gives the same bits each time, and matches the oracle."""
    wt, bias, _ = W.matmul_params()
    wt_d, bias_d = dev_bf16(wt), dev_bf16(bias)
    rng = np.random.default_rng(31)
    a = W.f32_to_bf16_bits((rng.standard_normal((3, 4096)) * 0.02).astype(np.float32))
    a_d = dev_bf16(a)
    ctx = D.Ctx(0)
    try:
        outs = []
        for _ in range(3):
            ctx.reset()
            out = ctx.feed(W.MATMUL_ABS_OPS, {"A": a_d, "W": wt_d.t(), "bias": bias_d}, ["y"])
            outs.append(host(out["y"]))
        img, _ = ctx.launch_log[-1]
        assert ctx.poll() == 0
    finally:
        ctx.close()
    tk = struct.unpack_from("<I", img, 48 + 24 + 16 + 8)[0]
    assert tk < 4096, "expected a K-split plan"
    assert np.array_equal(outs[0], outs[1]) and np.array_equal(outs[0], outs[2])
    check_bf16(outs[0], oracle_mm(a, wt, bias))


def test_matmul_identity_and_zero_are_exact():
    from oracle.bf16 import round_bf16
    rng = np.random.default_rng(9)
    n = 256
    a = W.f32_to_bf16_bits(rng.standard_normal((300, n)).astype(np.float32))
    eye = W.f32_to_bf16_bits(np.eye(n, dtype=np.float32))
    bias = W.f32_to_bf16_bits(rng.standard_normal(n).astype(np.float32))
    got = run_mm(dev_bf16(a), dev_bf16(eye).t(), dev_bf16(bias))
    ref = round_bf16(np.abs(bf16_bits_to_f64(a) + bf16_bits_to_f64(bias)[None, :]) * 0.5)
    assert np.array_equal(got, ref)
    zero = np.zeros_like(a)
    got0 = run_mm(dev_bf16(zero), dev_bf16(eye).t(), dev_bf16(bias))
    assert np.array_equal(got0, np.broadcast_to(round_bf16(np.abs(bf16_bits_to_f64(bias)) * 0.5), got0.shape))


def test_matmul_reproducible():
    wt, bias, _ = W.matmul_params()
    inp = W.matmul_inputs(1, 257, small_params=(wt, bias))
    a = dev_bf16(inp["A"][0])
    y1 = run_mm(a, dev_bf16(wt).t(), dev_bf16(bias))
    y2 = run_mm(a, dev_bf16(wt).t(), dev_bf16(bias))
    assert np.array_equal(y1, y2)


# ------------------------------------------------ other epilogue programs --
def test_matmul_epilogue_full_and_row_operands_fp32_out():
    """y = exp(-(A@W) * s) + r with s [M,N] fp32 and r [M,1] fp32: exercises full and
    per-row epilogue loads, a unary heavy op and an fp32 store."""
    ops = [
        ("matmul", ["A", "W"], "p", "f32", ()),
        ("mul", ["p", "s"], "q", "f32", ()),
        ("neg", ["q"], "q2", "f32", ()),
        ("exp", ["q2"], "e", "f32", ()),
        ("add", ["e", "r"], "y", "f32", ()),
    ]
    rng = np.random.default_rng(21)
    m, n, k = 190, 320, 256
    a = W.f32_to_bf16_bits((rng.standard_normal((m, k)) * 0.1).astype(np.float32))
    wt = W.f32_to_bf16_bits((rng.standard_normal((n, k)) * 0.1).astype(np.float32))
    s = rng.standard_normal((m, n)).astype(np.float32)
    r = rng.standard_normal((m, 1)).astype(np.float32)
    inputs = {"A": dev_bf16(a), "W": dev_bf16(wt).t(), "s": torch.from_numpy(s).cuda(),
              "r": torch.from_numpy(r).cuda()}
    ctx = D.Ctx(0)
    try:
        out = ctx.feed(ops, inputs, ["y"])
        assert ctx.poll() == 0
        kinds = [img[6] for img, _ in ctx.launch_log]
    finally:
        ctx.close()
    assert kinds == [2]
    got = host(out["y"])
    ref = evaluate(ops, {"A": (a, "bf16"), "W": (np.ascontiguousarray(wt.T), "bf16"), "s": (s, "f32"),
                         "r": (r, "f32")})["y"]
    err = np.abs(got - ref) / np.maximum(1.0, np.abs(ref))
    assert err.max() <= 1e-3, err.max()


# ------------------------------------------- addmm and the MatMul op alone --
def _run_one_cube_launch(ops, inputs, outs):
    ctx = D.Ctx(0)
    try:
        out = ctx.feed(ops, inputs, outs)
        assert ctx.poll() == 0
        kinds = [img[6] for img, _ in ctx.launch_log]
    finally:
        ctx.close()
    torch.cuda.synchronize()
    assert kinds == [2], "expected one CUBE launch, got kernel types %r" % kinds
    return {k: host(v) for k, v in out.items()}


@pytest.mark.parametrize("m", [1, 129, 300, 2048])
def test_addmm(m):
    """y = 2 * C + 0.5 * (A @ W): the beta-scaled full operand C is read by the epilogue."""
    wt, _, _ = W.matmul_params()
    inp = W.matmul_inputs(m, m, small_params=(wt, np.zeros(W.MM_N, np.uint16)))
    c = W.addmm_c(m, m)
    got = _run_one_cube_launch(W.ADDMM_OPS, {"A": dev_bf16(inp["A"][0]), "W": dev_bf16(wt).t(), "C": dev_bf16(c)},
                               W.ADDMM_OUT)["y"]
    ref = evaluate(W.ADDMM_OPS, {"A": inp["A"], "W": (np.ascontiguousarray(wt.T), "bf16"), "C": (c, "bf16")})["y"]
    check_bf16(got, ref)


@pytest.mark.parametrize("m,out_dt", [(1, "bf16"), (300, "bf16"), (129, "f32"), (1000, "f32"), (1, "f32"), (64, "f32")])
def test_matmul_alone(m, out_dt):
    """The MatMul op with no epilogue ops, bf16 or fp32 result; M = 1 and 64 run as
    K-split tiles (fp32 partials summed in split order), within the same fp32 bound."""
    wt, _, _ = W.matmul_params()
    inp = W.matmul_inputs(m + 1000, m, small_params=(wt, np.zeros(W.MM_N, np.uint16)))
    ops = [("matmul", ["A", "W"], "y", out_dt, ())]
    got = _run_one_cube_launch(ops, {"A": dev_bf16(inp["A"][0]), "W": dev_bf16(wt).t()}, ["y"])["y"]
    ref = evaluate(ops, {"A": inp["A"], "W": (np.ascontiguousarray(wt.T), "bf16")})["y"]
    if out_dt == "bf16":
        check_bf16(got, ref)
    else:
        # fp32 accumulation of K = 4096 exact bf16 products: the standard bound
        # gamma_K * sum_k |a_k w_k|, gamma_K = K u / (1 - K u), u = 2^-24
        a, w = bf16_bits_to_f64(inp["A"][0]), bf16_bits_to_f64(wt)
        k = a.shape[1]
        gamma = k * 2.0 ** -24 / (1 - k * 2.0 ** -24)
        assert np.all(np.abs(got - ref) <= gamma * (np.abs(a) @ np.abs(w).T) + 1e-30)


def test_matmul_dynamic_instances_sampled_rows():
    """Ten instances of the dynamic-M stream, each encoded as a new shape: 8 sampled
    rows per instance against the oracle."""
    wt, bias, _ = W.matmul_params()
    w_dev, b_dev = dev_bf16(wt).t(), dev_bf16(bias)
    ms = W.matmul_rows()[:10]
    for i, m in enumerate(ms):
        a = W.matmul_inputs(i, m, small_params=(wt, bias))["A"][0]
        got = run_mm(dev_bf16(a), w_dev, b_dev)
        rows = np.unique(np.random.default_rng(i).integers(0, m, 8))
        check_bf16(got[rows], oracle_mm(a[rows], wt, bias))
