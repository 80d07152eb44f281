"""fp64 -> bfloat16 rounding for the oracle (test infrastructure only).

bfloat16 keeps float32's 8 exponent bits and 7 stored mantissa bits, i.e. 8
significant bits.  Rounding is to nearest, ties to even, applied ONCE from the
exact fp64 value (the oracle never rounds through float32 first).  Overflow
follows IEEE 754 round-to-nearest: values at or above the midpoint between the
largest finite bfloat16 and 2**128 become +-inf.  Subnormal bfloat16 values
(down to 2**-133) are produced with the same spacing rule as float32
subnormals.  NaN stays NaN, +-inf and +-0 are kept.
"""
import numpy as np

_BF16_MAX = float.fromhex("0x1.fep127")          # largest finite bfloat16
_OVERFLOW_EDGE = float.fromhex("0x1.ffp127")     # midpoint to 2**128: ties go to even (= inf)
_MIN_NORMAL_EXP = -126                            # same exponent range as float32
_MANT_BITS = 8                                    # significant bits incl. the implicit one


def round_bf16(x):
    """Round an array of fp64 values to the nearest bfloat16 (ties to even).

    Returns fp64 values that are exactly representable in bfloat16.
    """
    x = np.asarray(x, dtype=np.float64)
    out = np.array(x, dtype=np.float64, copy=True)
    finite = np.isfinite(x) & (x != 0.0)
    v = x[finite]
    a = np.abs(v)
    # exponent e with 2**e <= |v| < 2**(e+1)
    _, e2 = np.frexp(a)               # a = m * 2**e2, 0.5 <= m < 1
    e = e2.astype(np.int64) - 1
    e = np.maximum(e, _MIN_NORMAL_EXP)  # below the normal range the spacing is fixed
    ulp_exp = e - (_MANT_BITS - 1)      # spacing of representable values at this exponent
    scaled = np.ldexp(a, -ulp_exp)      # exact: a power-of-two scaling
    r = np.rint(scaled)                 # numpy rint rounds half to even
    rounded = np.ldexp(r, ulp_exp)
    rounded = np.where(a >= _OVERFLOW_EDGE, np.inf, rounded)
    out[finite] = np.copysign(rounded, v)
    return out


def bf16_bits_to_f64(bits):
    """Exact value of bfloat16 bit patterns (uint16) as fp64."""
    b = np.asarray(bits, dtype=np.uint16).astype(np.uint32) << np.uint32(16)
    return b.view(np.float32).astype(np.float64)


def f64_to_bf16_bits(x):
    """Bit patterns of fp64 values that are already exact bfloat16 values."""
    f = np.asarray(x, dtype=np.float64).astype(np.float32)
    return (f.view(np.uint32) >> np.uint32(16)).astype(np.uint16)


BF16_MAX = _BF16_MAX
