"""Code-point tables and the BF16 rounding rule (oracle; test infrastructure only).

The pages name the formats but do not print their bit layouts:
  * "FP4 (E2M1, only 8 representable magnitudes)" -- MSLK PR #393,
    "Implementation Method";
  * E4M3 weights with float32 ``weight_scale_inv`` blocks -- transformers PR #50031,
    `_dequantize_fp8_weight`; E4M3 max 448 -- AstrAI fp8.py, FP8_MAX table;
  * E8M0 block scales (``float8_e8m0fnu``, group size 32) -- MindSpeed PR #3852,
    `MXFP8MatMul.forward`;
  * E5M2 for the gradient in the "hybrid" recipe (E4M3 forward, E5M2 backward), max
    57344 -- AstrAI fp8.py, `FP8Format` and the FP8_MAX table.
The layouts below are therefore taken from the public format definitions
(OCP 8-bit Floating Point Specification; OCP Microscaling Formats v1.0) and
written out code by code.
"""

import math

import numpy as np

# --------------------------------------------------------------------------
# E4M3 ("fn" flavour): 1 sign, 4 exponent (bias 7), 3 mantissa bits.
# exponent 0 is subnormal (m/8 * 2^-6); S.1111.111 is NaN; there is no infinity.
# --------------------------------------------------------------------------


def _e4m3_value(code: int) -> float:
    sign = -1.0 if (code >> 7) & 1 else 1.0
    exp = (code >> 3) & 0xF
    man = code & 0x7
    if exp == 0xF and man == 0x7:
        return math.nan
    if exp == 0:
        return sign * (man / 8.0) * 2.0 ** -6
    return sign * (1.0 + man / 8.0) * 2.0 ** (exp - 7)


E4M3_TABLE = np.array([_e4m3_value(c) for c in range(256)], dtype=np.float64)
E4M3_MAX = 448.0  # AstrAI fp8.py FP8_MAX["e4m3"]

# --------------------------------------------------------------------------
# E2M1: 1 sign, 2 exponent (bias 1), 1 mantissa bit; exponent 0 is subnormal (m * 0.5).
# --------------------------------------------------------------------------


def _e2m1_value(code: int) -> float:
    sign = -1.0 if (code >> 3) & 1 else 1.0
    exp = (code >> 1) & 0x3
    man = code & 0x1
    if exp == 0:
        return sign * man * 0.5
    return sign * (1.0 + man / 2.0) * 2.0 ** (exp - 1)


E2M1_TABLE = np.array([_e2m1_value(c) for c in range(16)], dtype=np.float64)

# --------------------------------------------------------------------------
# E8M0: unsigned power of two, byte b -> 2^(b-127); 0xFF is NaN.
# --------------------------------------------------------------------------


def _e8m0_value(b: int) -> float:
    if b == 0xFF:
        return math.nan
    return math.ldexp(1.0, b - 127)


E8M0_TABLE = np.array([_e8m0_value(b) for b in range(256)], dtype=np.float64)

# --------------------------------------------------------------------------
# E5M2: 1 sign, 5 exponent (bias 15), 2 mantissa bits; exponent 0 is subnormal
# (m/4 * 2^-14); exponent 31 is infinity (mantissa 0) or NaN (mantissa != 0).
# --------------------------------------------------------------------------


def _e5m2_value(code: int) -> float:
    sign = -1.0 if (code >> 7) & 1 else 1.0
    exp = (code >> 2) & 0x1F
    man = code & 0x3
    if exp == 0x1F:
        return math.nan if man else sign * math.inf
    if exp == 0:
        return sign * (man / 4.0) * 2.0 ** -14
    return sign * (1.0 + man / 4.0) * 2.0 ** (exp - 15)


E5M2_TABLE = np.array([_e5m2_value(c) for c in range(256)], dtype=np.float64)
E5M2_MAX = 57344.0  # AstrAI fp8.py FP8_MAX["e5m2"]


def e5m2_round(x):
    """E5M2 codes (uint8) of float64 values, rounded to the nearest E5M2 value, ties to
    the even code (mantissa bit 0 clear).

    Finite magnitudes beyond the largest finite value, and infinities, become +-57344
    (saturation to the finite range); NaN becomes the code 0x7F (sign kept); the sign
    of zero is kept.  The spacing of E5M2 values around |x| is 2^(floor(log2|x|) - 2)
    for normal magnitudes and 2^-16 below 2^-14, so rint(x / spacing) * spacing is the
    nearest-even value, as in bf16_round.
    """
    x = np.asarray(x, dtype=np.float64)
    ax = np.abs(x)
    finite = np.isfinite(ax) & (ax != 0)
    r = np.zeros_like(ax)
    _, e2 = np.frexp(ax[finite])
    expo = np.maximum(e2 - 1, -14)
    spacing = np.ldexp(1.0, expo - 2)
    r[finite] = np.rint(ax[finite] / spacing) * spacing
    r = np.where(np.isinf(ax) | (r > E5M2_MAX), E5M2_MAX, r)
    # value -> code: the table's positive codes 0x00..0x7B hold every finite magnitude
    # in increasing order
    codes = np.searchsorted(E5M2_TABLE[:0x7C], r).astype(np.uint8)
    codes = np.where(np.signbit(x), codes | 0x80, codes).astype(np.uint8)
    return np.where(np.isnan(x), np.where(np.signbit(x), 0xFF, 0x7F), codes).astype(np.uint8)


# --------------------------------------------------------------------------
# BF16 round-to-nearest-even from an exact float64 value.
# BF16 = 1 sign, 8 exponent (bias 127), 7 mantissa bits; subnormals kept.
# --------------------------------------------------------------------------

_BF16_MIN_NORMAL_EXP = -126
_BF16_MAN_BITS = 7


def bf16_round(x):
    """Round float64 values to the nearest BF16 value, ties to even.

    Works on the exact float64 input: the spacing of BF16 values around |x| is
    2^(floor(log2|x|) - 7) for normal magnitudes and 2^-133 below 2^-126, so
    rint(x / spacing) * spacing is the nearest-even BF16 value (np.rint rounds
    half to even, and x / spacing is exact because spacing is a power of two).
    Values whose rounded magnitude reaches 2^128 become infinities.  NaN stays
    NaN.  The sign of zero is kept.
    """
    x = np.asarray(x, dtype=np.float64)
    out = np.array(x, dtype=np.float64, copy=True)
    finite = np.isfinite(x) & (x != 0)
    ax = np.abs(x[finite])
    _, e2 = np.frexp(ax)  # ax = m * 2^e2 with m in [0.5, 1)  =>  floor(log2 ax) = e2 - 1
    expo = np.maximum(e2 - 1, _BF16_MIN_NORMAL_EXP)
    spacing = np.ldexp(1.0, expo - _BF16_MAN_BITS)
    r = np.rint(ax / spacing) * spacing
    r = np.where(r >= 2.0 ** 128, np.inf, r)
    out[finite] = np.copysign(r, x[finite])
    return out


def bf16_bits(x):
    """BF16 bit patterns (uint16) of float64 values that are already BF16 values.

    NaNs map to the canonical quiet NaN 0x7FC0 (sign kept); comparisons treat
    every NaN pattern as one class.
    """
    x = np.asarray(x, dtype=np.float64)
    f32 = x.astype(np.float32)  # exact: every BF16 value is a float32 value
    bits = (f32.view(np.uint32) >> 16).astype(np.uint16)
    nan = np.isnan(x)
    if nan.any():
        bits = bits.copy()
        bits[nan] = np.where(np.signbit(x[nan]), 0xFFC0, 0x7FC0).astype(np.uint16)
    return bits


def bf16_from_bits(bits):
    """float64 values of BF16 bit patterns (uint16)."""
    bits = np.asarray(bits, dtype=np.uint16)
    return (bits.astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def bf16_is_nan_bits(bits):
    bits = np.asarray(bits, dtype=np.uint16)
    return ((bits & 0x7F80) == 0x7F80) & ((bits & 0x007F) != 0)


def fp32_round(x):
    """Round exact float64 values to float32 (IEEE nearest-even, subnormals kept)."""
    return np.asarray(x, dtype=np.float64).astype(np.float32).astype(np.float64)
