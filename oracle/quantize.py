"""Per-tensor E5M2 quantization of a gradient (oracle; test infrastructure only).

AstrAI fp8.py, `_LinearFp8.backward` and the recipe classes: in the "hybrid" format the
backward quantizes the incoming gradient once to E5M2, and both products (dX, dW) use
that one quantization.  The quantization step of a tensor is

    step = (amax / FP8_MAX["e5m2"]) / 2^margin,    FP8_MAX["e5m2"] = 57344,

where, under dynamic scaling, amax is the current tensor's max |value| taken in float32
and clamped below at 1e-12 (`_dynamic_scale`, `DynamicScaling.scale_from_history`).

Readings taken where the pages say nothing (the quantizing kernel itself is not shown):
  * quantized value = gradient / step, one IEEE float32 division, then rounded to the
    nearest E5M2 value, ties to even, with finite saturation (formats.e5m2_round);
  * amax of a tensor holding a NaN is NaN (torch's amax propagates it), so every code
    is then NaN.

Shapes: any; the gradient is given as float64 values that are BF16 numbers.
"""

import numpy as np

from .formats import E5M2_MAX, e5m2_round, fp32_round

AMAX_FLOOR = 1e-12  # `_dynamic_scale`: amax.clamp_min(1e-12)


def amax_f32(g):
    """max |g| as a float32 value (float64 holder), NaN if g holds a NaN, at least 1e-12."""
    g = np.asarray(g, dtype=np.float64)
    a = np.max(np.abs(g)) if g.size else 0.0
    if np.isnan(a):
        return float("nan")
    return float(max(fp32_round(a), fp32_round(AMAX_FLOOR)))


def e5m2_step(amax, margin=0):
    """The quantization step (amax / 57344) / 2^margin, each division in float32."""
    return float(fp32_round(fp32_round(amax / E5M2_MAX) / 2.0 ** margin))


def quantize_e5m2(g, margin=0):
    """(codes uint8, step, amax) of the dynamic per-tensor E5M2 quantization of g."""
    g = np.asarray(g, dtype=np.float64)
    amax = amax_f32(g)
    step = e5m2_step(amax, margin)
    q = fp32_round(g / step)   # float32 division: the quotient of two float32 values, rounded once
    return e5m2_round(q), step, amax
