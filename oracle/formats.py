"""Number formats: E4M3 (finite-number "fn" variant) and BF16.

Oracle module (test infrastructure only).

The pages fix E4M3 as 4 exponent bits and 3 mantissa bits with largest finite value
448, smallest normal 1.562e-2 (= 2**-6) and 8 steps per octave ("DeepSeek-V3: the
recipe, and the interconnect that shaped it", format table in "FP8: the other half of
the byte reduction"), used for every FP8 tensor ("DeepSeek-V3", core idea 6(c)), in
the finite-number convention (DeepSeek-V3 book, ch. 16 "Exponent and mantissa").

Reading taken where the pages are silent: rounding is round-to-nearest-even; a value
beyond 448 saturates to +-448 (the fn variant has no infinity); NaN encodes as 0x7F;
the sign of a zero result is kept (0x80 is -0).  Subnormals have exponent field 0 and
unit 2**-9.
"""

import numpy as np

E4M3_MAX = 448.0
E4M3_MIN_NORMAL = 2.0 ** -6      # exponent field 1, bias 7
E4M3_FRAC_BITS = 3
E4M3_SUBNORMAL_UNIT = 2.0 ** -9  # 2**(1 - 7 - 3)

BF16_FRAC_BITS = 7
BF16_MIN_NORMAL_EXP = -126
BF16_MAX = (2.0 - 2.0 ** -7) * 2.0 ** 127


def _round_binary(a, frac_bits, min_normal_exp):
    """Round non-negative float64 ``a`` to the nearest value with ``frac_bits``
    fraction bits (ties to even), using the subnormal grid below 2**min_normal_exp.

    frexp gives a = m * 2**ex with m in [0.5, 1), so the unbiased exponent is ex - 1.
    Dividing by the quantum (a power of two) is exact, and np.rint rounds half to even.
    """
    _, ex = np.frexp(a)
    e = np.maximum(ex - 1, min_normal_exp)
    quantum = np.ldexp(1.0, e - frac_bits)
    return np.rint(a / quantum) * quantum


def e4m3_round(v):
    """Value of ``v`` (float32 or float64 array) after RNE + saturating E4M3 rounding.

    Returns float64; NaN stays NaN, +-inf saturate to +-448 like any out-of-range value.
    """
    v = np.asarray(v, dtype=np.float64)
    with np.errstate(invalid="ignore"):
        a = np.abs(v)
        finite = np.isfinite(a)
        q = _round_binary(np.where(finite, a, 0.0), E4M3_FRAC_BITS, -6)
        q = np.where(finite, q, np.where(np.isnan(a), np.nan, E4M3_MAX))
        q = np.minimum(q, E4M3_MAX)
        q = np.where(np.isnan(a), np.nan, q)
    return np.copysign(q, v)


def e4m3_encode(v):
    """Encode float values to E4M3 bytes (uint8), RNE, saturating, NaN -> 0x7F."""
    v = np.asarray(v)
    q = e4m3_round(v)
    nan = np.isnan(q)
    a = np.abs(np.where(nan, 0.0, q))
    sign = np.signbit(np.where(nan, 0.0, q)).astype(np.uint8)
    normal = a >= E4M3_MIN_NORMAL
    _, ex = np.frexp(np.where(normal, a, 1.0))
    e = ex - 1                                   # unbiased exponent, -6 .. 8
    mant_normal = np.rint((np.where(normal, a, 1.0) / np.ldexp(1.0, e) - 1.0) * 8.0)
    code_normal = ((e + 7).astype(np.int64) << 3) | mant_normal.astype(np.int64)
    code_sub = np.rint(a / E4M3_SUBNORMAL_UNIT).astype(np.int64)   # 0 .. 7
    code = np.where(normal, code_normal, code_sub) | (sign.astype(np.int64) << 7)
    code = np.where(nan, 0x7F, code)
    return code.astype(np.uint8)


def e4m3_decode_table():
    """float64[256]: the value of every E4M3 code, from the bit definition (bias 7)."""
    t = np.empty(256, dtype=np.float64)
    for c in range(256):
        sign = -1.0 if c & 0x80 else 1.0
        exp_field = (c >> 3) & 0xF
        mant = c & 0x7
        if exp_field == 0xF and mant == 0x7:
            t[c] = np.nan
        elif exp_field == 0:
            t[c] = sign * mant * E4M3_SUBNORMAL_UNIT
        else:
            t[c] = sign * (1.0 + mant / 8.0) * 2.0 ** (exp_field - 7)
    return t


_DECODE = e4m3_decode_table()


def e4m3_decode(codes):
    """Decode uint8 E4M3 codes to float64."""
    return _DECODE[np.asarray(codes, dtype=np.uint8)]


def bf16_round(v):
    """Round float32/float64 values to BF16 (RNE, overflow to inf); returns float32.

    BF16 has 8 significant bits and the float32 exponent range.
    """
    v = np.asarray(v, dtype=np.float64)
    with np.errstate(invalid="ignore", over="ignore"):
        a = np.abs(v)
        finite = np.isfinite(a)
        q = _round_binary(np.where(finite, a, 0.0), BF16_FRAC_BITS, BF16_MIN_NORMAL_EXP)
        q = np.where(q > BF16_MAX, np.inf, q)
        q = np.where(finite, q, a)
    return np.copysign(q, v).astype(np.float32)
