"""Seeded synthetic workloads: input draws and the op streams fed to the fuser.

This module holds no arithmetic of the method.  It draws inputs (numpy on the
host for parity tests, torch on the device for the benchmark pools) and states
each workload's op stream as plain data: tuples of
(op, input_names, out_name, out_dtype, attrs).  Both the CUDA path (through
`bytecode_vm_jit_gb300.Ctx`) and the oracle consume these tuples.

Workloads (synthetic stand-ins for the DVM review page's Table 3 operators
and the Qwen3-14B fine-tuning run in the MindSpore DVM summary, section 4.3):

  sqrt_add     c = sqrt(a + b), fp32 4096x1024, U[0,1), seed 0, one shape
  layernorm    LayerNorm over 4096, fp32, R = B*S rows, B~U{1..32},
               S~U{1..2048}, 200 instances, seed 1, gamma~N(1,.1), beta~N(0,.1)
  if_else_add  y = x+z if sum(x) > 0 else x-z, bf16 [T,8192], T~U{64..16384},
               500 instances, seed 2, branches forced by sign-flipping x
  matmul_abs   y = |A @ W + bias| * 0.5, bf16 in / fp32 acc / bf16 out,
               A[M,4096], W[4096,4096] (stored as Wt[N,K], K contiguous),
               M log-uniform in [1,8192], 100 instances, seed 3
  qwen_stream  per step h = x + r; n = RMSNorm(h)*w (eps 1e-6);
               s = silu(g)*u; hidden 5120, intermediate 17408,
               T~U{128..4096}, 2000 steps, seed 4

Conventions: a bf16 array is carried as its uint16 bit patterns in numpy and
as torch.bfloat16 on the device; fp32 -> bf16 conversion of drawn values is
torch's round-to-nearest-even.
"""
import math

import numpy as np

HIDDEN = 5120
INTER = 17408
LN_D = 4096
IEA_D = 8192
MM_K = 4096
MM_N = 4096

# --------------------------------------------------------------------------
# op streams (data only)
# --------------------------------------------------------------------------
SQRT_ADD_OPS = [
    ("add", ["a", "b"], "c", "f32", ()),
    ("sqrt", ["c"], "y", "f32", ()),
]
SQRT_ADD_OUT = ["y"]

LAYERNORM_EPS = 1e-5
LAYERNORM_OPS = [
    ("reduce_mean", ["x"], "mu", "f32", ()),
    ("sub", ["x", "mu"], "xc", "f32", ()),
    ("mul", ["xc", "xc"], "sq", "f32", ()),
    ("reduce_mean", ["sq"], "var", "f32", ()),
    ("adds", ["var"], "ve", "f32", (LAYERNORM_EPS, 0)),
    ("pows", ["ve"], "rstd", "f32", (-0.5, 0)),
    ("mul", ["xc", "rstd"], "xn", "f32", ()),
    ("mul", ["xn", "gamma"], "xg", "f32", ()),
    ("add", ["xg", "beta"], "y", "f32", ()),
]
LAYERNORM_OUT = ["y"]

IF_ELSE_ADD_OPS = [
    ("reduce_sum_all", ["x"], "s", "f32", ()),
    ("add", ["x", "z"], "t", "bf16", ()),
    ("sub", ["x", "z"], "e", "bf16", ()),
    ("select_gt0", ["s", "t", "e"], "y", "bf16", ()),
]
IF_ELSE_ADD_OUT = ["y"]
# host-sync variant: the predicate is materialised, read on the host, and only
# the chosen branch op is captured afterwards
IF_ELSE_PRED_OPS = [("reduce_sum_all", ["x"], "s", "f32", ())]
IF_ELSE_THEN_OPS = [("add", ["x", "z"], "y", "bf16", ())]
IF_ELSE_ELSE_OPS = [("sub", ["x", "z"], "y", "bf16", ())]

MATMUL_ABS_OPS = [
    ("matmul", ["A", "W"], "p", "f32", ()),
    ("add", ["p", "bias"], "q", "f32", ()),
    ("abs", ["q"], "r", "f32", ()),
    ("muls", ["r"], "y", "bf16", (0.5, 0)),
]
MATMUL_ABS_OUT = ["y"]

# addmm (the review's Table 3 op): y = beta * C + alpha * (A @ W), C a full [M, N]
# operand read by the epilogue; and the MatMul tile op alone (bf16 result)
ADDMM_ALPHA, ADDMM_BETA = 0.5, 2.0
ADDMM_OPS = [
    ("matmul", ["A", "W"], "p", "f32", ()),
    ("muls", ["p"], "q", "f32", (ADDMM_ALPHA, 0)),
    ("muls", ["C"], "c2", "f32", (ADDMM_BETA, 0)),
    ("add", ["q", "c2"], "y", "bf16", ()),
]
ADDMM_OUT = ["y"]
MATMUL_OPS = [("matmul", ["A", "W"], "y", "bf16", ())]
MATMUL_OUT = ["y"]

RMS_EPS = 1e-6
QWEN_STEP_OPS = [
    ("add", ["x", "r"], "h", "bf16", ()),
    ("mul", ["h", "h"], "h2", "f32", ()),
    ("reduce_mean", ["h2"], "ms", "f32", ()),
    ("adds", ["ms"], "mse", "f32", (RMS_EPS, 0)),
    ("pows", ["mse"], "rs", "f32", (-0.5, 0)),
    ("mul", ["h", "rs"], "hn", "f32", ()),
    ("mul", ["hn", "w"], "n", "bf16", ()),
    ("silu", ["g"], "sg", "f32", ()),
    ("mul", ["sg", "u"], "s", "bf16", ()),
    # stands for the step's ops DVM does not run (projections, attention, ...)
    ("opaque", [], "", "f32", ()),
]
QWEN_STEP_OUT = ["h", "n", "s"]


# --------------------------------------------------------------------------
# draws
# --------------------------------------------------------------------------
def f32_to_bf16_bits(a):
    """bfloat16 bit patterns (uint16) of float32 data, round-to-nearest-even."""
    import torch
    t = torch.from_numpy(np.ascontiguousarray(a, dtype=np.float32)).to(torch.bfloat16)
    return t.view(torch.int16).numpy().view(np.uint16)


def bf16_bits_to_torch(bits):
    import torch
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(torch.bfloat16)


def _normal_f32(rng, shape, mean=0.0, std=1.0):
    x = rng.standard_normal(shape, dtype=np.float32)
    if std != 1.0:
        x *= np.float32(std)
    if mean != 0.0:
        x += np.float32(mean)
    return x


# sqrt_add ------------------------------------------------------------------
def sqrt_add_inputs(shape=(4096, 1024), seed=0):
    rng = np.random.default_rng(seed)
    a = rng.random(shape, dtype=np.float32)
    b = rng.random(shape, dtype=np.float32)
    return {"a": (a, "f32"), "b": (b, "f32")}


# layernorm -----------------------------------------------------------------
def layernorm_params(seed=1, d=LN_D):
    rng = np.random.default_rng(seed)
    gamma = _normal_f32(rng, (d,), 1.0, 0.1)
    beta = _normal_f32(rng, (d,), 0.0, 0.1)
    return gamma, beta, rng


def layernorm_rows(n=200, seed=1):
    """Row counts R = B*S of the dynamic instances (B~U{1..32}, S~U{1..2048})."""
    _, _, rng = layernorm_params(seed)
    rows = []
    for _ in range(n):
        b = int(rng.integers(1, 33))
        s = int(rng.integers(1, 2049))
        rows.append(b * s)
    return rows


def layernorm_inputs(i, rows, seed=1, d=LN_D):
    gamma, beta, _ = layernorm_params(seed, d)
    rng = np.random.default_rng([seed, i])
    x = _normal_f32(rng, (rows, d))
    return {"x": (x, "f32"), "gamma": (gamma, "f32"), "beta": (beta, "f32")}


# if_else_add -----------------------------------------------------------------
def if_else_rows(n=500, seed=2):
    rng = np.random.default_rng(seed)
    return [int(rng.integers(64, 16385)) for _ in range(n)]


def if_else_inputs(i, rows, seed=2, d=IEA_D):
    """x, z ~ N(0,1) in bf16; instance i even wants sum(x) > 0, odd wants <= 0.

    The sign of x is flipped (exactly) when the fp64 sum of the bf16 values has
    the wrong sign.
    """
    rng = np.random.default_rng([seed, i])
    xb = f32_to_bf16_bits(_normal_f32(rng, (rows, d)))
    zb = f32_to_bf16_bits(_normal_f32(rng, (rows, d)))
    xs = (xb.astype(np.uint32) << np.uint32(16)).view(np.float32)
    s = float(np.sum(xs, dtype=np.float64))
    want_pos = (i % 2 == 0)
    if (s > 0) != want_pos:
        xb = xb ^ np.uint16(0x8000)
    return {"x": (xb, "bf16"), "z": (zb, "bf16")}


# matmul_abs ------------------------------------------------------------------
def matmul_params(seed=3, k=MM_K, n=MM_N):
    rng = np.random.default_rng(seed)
    wt = f32_to_bf16_bits(_normal_f32(rng, (n, k), 0.0, 0.02))   # Wt[N,K]
    bias = f32_to_bf16_bits(_normal_f32(rng, (n,), 0.0, 0.1))
    return wt, bias, rng


def matmul_rows(n=100, seed=3):
    rng = np.random.default_rng([seed, 1 << 20])
    out = []
    for _ in range(n):
        u = float(rng.random())
        out.append(min(8192, max(1, int(math.floor(math.exp(u * math.log(8193)))))))
    return out


def matmul_inputs(i, m, seed=3, k=MM_K, n=MM_N, small_params=None):
    if small_params is None:
        wt, bias, _ = matmul_params(seed, k, n)
    else:
        wt, bias = small_params
    rng = np.random.default_rng([seed, i])
    a = f32_to_bf16_bits(_normal_f32(rng, (m, k), 0.0, 0.02))
    return {"A": (a, "bf16"), "Wt": (wt, "bf16"), "bias": (bias, "bf16")}


def addmm_c(i, m, seed=5, n=MM_N):
    """C [m, n] bf16 ~ N(0, 0.1) for instance i."""
    rng = np.random.default_rng([seed, i])
    return f32_to_bf16_bits(_normal_f32(rng, (m, n), 0.0, 0.1))


# qwen_stream -----------------------------------------------------------------
def qwen_weight(seed=4, hidden=HIDDEN):
    rng = np.random.default_rng(seed)
    w = f32_to_bf16_bits(_normal_f32(rng, (hidden,), 1.0, 0.02))
    return w, rng


def qwen_tokens(n=2000, seed=4):
    _, rng = qwen_weight(seed)
    return [int(rng.integers(128, 4097)) for _ in range(n)]


def qwen_inputs(i, t, seed=4, hidden=HIDDEN, inter=INTER):
    w, _ = qwen_weight(seed, hidden)
    rng = np.random.default_rng([seed, i])
    x = f32_to_bf16_bits(_normal_f32(rng, (t, hidden)))
    r = f32_to_bf16_bits(_normal_f32(rng, (t, hidden)))
    g = f32_to_bf16_bits(_normal_f32(rng, (t, inter)))
    u = f32_to_bf16_bits(_normal_f32(rng, (t, inter)))
    return {"x": (x, "bf16"), "r": (r, "bf16"), "w": (w, "bf16"),
            "g": (g, "bf16"), "u": (u, "bf16")}


# --------------------------------------------------------------------------
# device pools for the benchmark (torch, seeded; values are N(0,1) or U[0,1))
# --------------------------------------------------------------------------
def device_pool(nbytes, dtype, dist, seed, device="cuda", std=1.0):
    """A flat device tensor of about `nbytes` bytes drawn from a seeded generator
    (normal draws are scaled by `std` in fp32 before the cast)."""
    import torch
    tdt = {"f32": torch.float32, "bf16": torch.bfloat16}[dtype]
    esz = 4 if dtype == "f32" else 2
    n = int(nbytes) // esz
    g = torch.Generator(device=device)
    g.manual_seed(int(seed))
    out = torch.empty(n, dtype=tdt, device=device)
    chunk = 1 << 27
    for o in range(0, n, chunk):
        m = min(chunk, n - o)
        if dist == "normal":
            out[o:o + m] = (torch.randn(m, generator=g, device=device, dtype=torch.float32) * std).to(tdt)
        else:
            out[o:o + m] = torch.rand(m, generator=g, device=device, dtype=torch.float32).to(tdt)
    return out
