"""Op-graph evaluator: the oracle for every fused program (test infrastructure).

What the DVM path computes is the eager op stream that the streaming fuser
captures (DVM review page, section 5.2 "dynamic graph fusion"; MindSpore DVM
summary, section 3.2): each captured op has a value semantics of its own and
fusion must not change it beyond rounding.  This evaluator therefore runs the
op list one op at a time, with no bytecode, tiling or fusion:

* every input value is taken exactly (bfloat16 inputs are widened bit-exactly);
* the op is computed in fp64 (numpy);
* the result is rounded ONCE to the op's declared output dtype
  (float32: IEEE round-to-nearest-even; bfloat16: `oracle.bf16.round_bf16`;
  uint8: the 0/1 predicate value).

Op semantics (DVM review page, Table 1 "tile-level virtual instructions", plus
the binary/reduce/matmul ops its fusion patterns need -- section 5.1 names
c = a + b, the vector-vector example, and cube-vector matmul fusion; the
MindSpore summary, section 3.3, names Elemwise, Reduce-forward and
MatMul+Elemwise patterns):

  sqrt abs log exp round floor isfinite neg rsqrt recip silu copy cast
  add sub mul div max min pow            numpy broadcasting of two tensors
  adds subs muls divs maxs mins pows     tensor with a float32 scalar attribute;
                                         attrs = (scalar, left) -- left=1 puts the
                                         scalar on the left (s - x, s / x, s ** x)
  reduce_sum reduce_max reduce_mean      over the last axis, keepdims
  reduce_sum_all                         over every element, result shape (1,)
  select_gt0(p, a, b)                    a where the scalar p > 0, else b
                                         (NaN selects b)
  matmul(A, W)                           A[M,K] @ W[K,N]
  opaque                                 an op DVM does not run; evaluates nothing

Readings of points the pages leave open (each listed in the design notes):
round = half to even; max/min propagate NaN; log(0) = -inf, log(<0) = NaN;
pow follows C99 (negative base with non-integer exponent = NaN); isfinite
yields 1/0 in uint8; reduce_mean = exact sum / n; rsqrt = 1/sqrt(x);
silu(x) = x / (1 + exp(-x)).
"""
import numpy as np

from .bf16 import round_bf16, bf16_bits_to_f64

DTYPES = ("f32", "bf16", "u8")

UNARY = {
    "sqrt": np.sqrt,
    "abs": np.abs,
    "log": np.log,
    "exp": np.exp,
    "round": np.rint,
    "floor": np.floor,
    "neg": np.negative,
    "rsqrt": lambda x: 1.0 / np.sqrt(x),
    "recip": lambda x: 1.0 / x,
    "silu": lambda x: x / (1.0 + np.exp(-x)),
    "copy": lambda x: x,
    "cast": lambda x: x,
    "isfinite": lambda x: np.isfinite(x).astype(np.float64),
}

BINARY = {
    "add": np.add,
    "sub": np.subtract,
    "mul": np.multiply,
    "div": np.divide,
    "max": np.maximum,
    "min": np.minimum,
    "pow": np.power,
}

SCALAR = {k + "s": v for k, v in BINARY.items() if k != "pow"}
SCALAR["pows"] = np.power


def round_to(x, dtype):
    """Round fp64 values once to `dtype`; returns fp64 holding the rounded values."""
    x = np.asarray(x, dtype=np.float64)
    if dtype == "f32":
        return x.astype(np.float32).astype(np.float64)
    if dtype == "bf16":
        return round_bf16(x)
    if dtype == "u8":
        return x
    raise ValueError("unknown dtype %r" % (dtype,))


def as_f64(arr, dtype):
    """Exact fp64 value of an input array given in its storage form.

    float32 arrays are widened; bfloat16 data is given as uint16 bit patterns;
    uint8 arrays are widened.
    """
    if dtype == "bf16":
        return bf16_bits_to_f64(arr)
    return np.asarray(arr).astype(np.float64)


def eval_op(op, args, dtype, attrs=()):
    """Evaluate one op on fp64 arguments; return the rounded fp64 result."""
    with np.errstate(all="ignore"):
        if op in UNARY:
            (x,) = args
            r = UNARY[op](x)
        elif op in BINARY:
            a, b = args
            r = BINARY[op](a, b)
        elif op in SCALAR:
            (x,) = args
            s = float(np.float32(attrs[0]))
            left = len(attrs) > 1 and attrs[1] != 0
            r = SCALAR[op](s, x) if left else SCALAR[op](x, s)
        elif op == "reduce_sum":
            (x,) = args
            r = np.sum(x, axis=-1, keepdims=True)
        elif op == "reduce_max":
            (x,) = args
            r = np.max(x, axis=-1, keepdims=True)
        elif op == "reduce_mean":
            (x,) = args
            r = np.sum(x, axis=-1, keepdims=True) / x.shape[-1]
        elif op == "reduce_sum_all":
            (x,) = args
            r = np.array([np.sum(x)])
        elif op == "select_gt0":
            p, a, b = args
            r = np.array(a if p.reshape(-1)[0] > 0 else b, dtype=np.float64)
        elif op == "matmul":
            a, w = args
            r = np.matmul(a, w)
        elif op == "broadcast":
            (x,) = args
            r = np.broadcast_to(x, tuple(int(v) for v in attrs)).copy()
        else:
            raise ValueError("unknown op %r" % (op,))
    return round_to(r, dtype)


def evaluate(ops, inputs):
    """Run an op list.

    ops    : sequence of (op, input_names, out_name, out_dtype, attrs)
    inputs : dict name -> (array in storage form, dtype)
    returns: dict name -> fp64 array for every input and every op result
    """
    env = {name: as_f64(arr, dt) for name, (arr, dt) in inputs.items()}
    for op, ins, out, dtype, attrs in ops:
        if op == "opaque":
            continue
        env[out] = eval_op(op, [env[n] for n in ins], dtype, attrs)
    return env
