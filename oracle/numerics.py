"""Number formats used by the oracle: bf16 (as uint16 bits) and fp8 e4m3.

TEST INFRASTRUCTURE (see the package docstring).

bf16 is the top half of an IEEE-754 binary32: 1 sign bit, 8 exponent bits
(bias 127), 7 fraction bits. Decoding is exact (shift the 16 bits into the high
half of a binary32). Encoding rounds a float64 to the nearest bf16 with ties to
even, written from the definition of round-to-nearest-even on the value, not by
bit tricks on a float32, so that no double rounding through float32 happens.

fp8 e4m3 ("e4m3fn") is 1 sign bit, 4 exponent bits (bias 7), 3 fraction bits;
exponent 0 holds subnormals, ``S.1111.111`` is NaN, there is no infinity, and
the largest finite magnitude is 448. The pages name the format only ("FP8 PLE
table", PR#54371 report 实现拆解 item 1; PR#53899 page, FP8 checkpoint
report); its bit layout is the OCP FP8 definition.
"""

import math

import numpy as np

# Largest finite bf16: (2 - 2^-7) * 2^127.
_BF16_MAX = (2.0 - 2.0 ** -7) * 2.0 ** 127
# Smallest positive normal bf16 and the quantum of the subnormal range.
_BF16_MIN_NORMAL = 2.0 ** -126
_BF16_SUBNORMAL_QUANTUM = 2.0 ** -133


def bf16_bits_to_f64(bits):
    """Exact value of bf16 bit patterns (uint16 array) as float64."""
    b = np.asarray(bits, dtype=np.uint16).astype(np.uint32) << np.uint32(16)
    return b.view(np.float32).astype(np.float64)


def _round_half_even_to_bf16_value(x):
    """Nearest bf16 value (ties to even) of finite float64 ``x``, as float64.

    Normal range: |x| = m * 2^e with m in [0.5, 1); bf16 keeps 8 significant
    bits, so the representable neighbours are multiples of 2^(e-8). numpy's
    ``rint`` rounds half to even and is exact here because m * 2^8 is an exact
    float64. A carry to 2^e needs no special case. Subnormal range: the
    quantum is fixed at 2^-133. Overflow past the largest finite bf16 plus half
    an ulp goes to infinity (the IEEE rule).
    """
    x = np.asarray(x, dtype=np.float64)
    out = np.empty_like(x)
    ax = np.abs(x)
    normal = ax >= _BF16_MIN_NORMAL
    m, e = np.frexp(x[normal])
    out[normal] = np.ldexp(np.rint(np.ldexp(m, 8)), e - 8)
    sub = ~normal
    out[sub] = np.rint(x[sub] / _BF16_SUBNORMAL_QUANTUM) * _BF16_SUBNORMAL_QUANTUM
    # Overflow threshold: halfway between max finite and 2^128 rounds to even,
    # which is the infinity side (max finite has an odd last bit).
    over = np.abs(out) > _BF16_MAX
    out[over] = np.copysign(np.inf, x[over])
    return out


def f64_to_bf16_bits(x):
    """Round float64 values to bf16 (nearest, ties to even); return uint16 bits.

    NaN maps to a quiet NaN with the input's sign (0x7FC0 / 0xFFC0).
    """
    x = np.asarray(x, dtype=np.float64)
    shape = x.shape
    flat = x.reshape(-1)
    nan = np.isnan(flat)
    vals = np.where(nan, 0.0, flat)
    inf = np.isinf(vals)
    r = np.empty_like(vals)
    r[inf] = vals[inf]
    r[~inf] = _round_half_even_to_bf16_value(vals[~inf])
    # r now holds values exactly representable in bf16 (hence in float32):
    # the float32 conversion is exact and its high half is the bf16 pattern.
    bits = (r.astype(np.float32).view(np.uint32) >> np.uint32(16)).astype(np.uint16)
    sign = np.signbit(flat)
    bits[nan] = np.where(sign[nan], 0xFFC0, 0x7FC0).astype(np.uint16)
    return bits.reshape(shape)


def e4m3_code_to_float(code):
    """Value of one fp8 e4m3 code (0..255) as a Python float (NaN for NaN)."""
    code = int(code) & 0xFF
    sign = -1.0 if code & 0x80 else 1.0
    exponent = (code >> 3) & 0xF
    fraction = code & 0x7
    if exponent == 0xF and fraction == 0x7:
        return math.nan
    if exponent == 0:
        # subnormal: 0.fff * 2^(1 - bias)
        return sign * (fraction / 8.0) * 2.0 ** (1 - 7)
    return sign * (1.0 + fraction / 8.0) * 2.0 ** (exponent - 7)


# Every code's value; all are exact in float32 (at most 4 significant bits).
E4M3_VALUES = np.array([e4m3_code_to_float(c) for c in range(256)], dtype=np.float32)
