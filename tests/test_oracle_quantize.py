"""Pins of the E5M2 gradient quantization oracle (oracle/quantize.py, formats.E5M2_*).

What fixes each piece, other than the oracle itself:
  * the E5M2 code table: torch's float8_e5m2 decoding of all 256 codes, and closed forms
    (the AstrAI page's maximum 57344, smallest subnormal 2^-16, smallest normal 2^-14,
    infinities and NaNs);
  * rounding to E5M2: torch's float32 -> float8_e5m2 cast on random values across the
    whole range and on every midpoint between neighbouring codes (ties to even), plus
    saturation beyond the range;
  * the quantizer: the AstrAI recipe written with torch ops (max |g| in float32 clamped
    at 1e-12, step = amax / 57344, g / step cast to float8_e5m2), the largest element
    landing on +-57344, the all-zero and NaN special cases;
  * the dequantization of E5M2 codes with a per-tensor step: torch's BF16 product of the
    code and the step cast to BF16.
"""

import numpy as np
import pytest
import torch

from oracle import dequant as D
from oracle import formats as F
from oracle import quantize as Q


def _torch_codes(x):
    """float8_e5m2 codes of float64 values through torch's float32 cast."""
    return torch.from_numpy(np.asarray(x, dtype=np.float32)).to(torch.float8_e5m2).view(torch.uint8).numpy()


def _same_codes(a, b):
    """Equal codes, every NaN code (exponent 31, mantissa != 0) one class."""
    nan = lambda c: ((c & 0x7C) == 0x7C) & ((c & 0x03) != 0)
    a, b = np.asarray(a, dtype=np.uint8), np.asarray(b, dtype=np.uint8)
    return np.array_equal(nan(a), nan(b)) and np.array_equal(a[~nan(a)], b[~nan(b)])


def test_e5m2_table_matches_torch_float8():
    t = torch.arange(256, dtype=torch.uint8).view(torch.float8_e5m2).double().numpy()
    a = F.E5M2_TABLE
    assert np.array_equal(np.isnan(a), np.isnan(t))
    assert np.array_equal(a[~np.isnan(a)], t[~np.isnan(t)])


def test_e5m2_closed_forms():
    assert F.E5M2_MAX == 57344.0 == F.E5M2_TABLE[0x7B] == -F.E5M2_TABLE[0xFB]
    assert F.E5M2_TABLE[0x01] == 2.0 ** -16 and F.E5M2_TABLE[0x04] == 2.0 ** -14
    assert F.E5M2_TABLE[0x7C] == np.inf and F.E5M2_TABLE[0xFC] == -np.inf
    assert all(np.isnan(F.E5M2_TABLE[c]) for c in (0x7D, 0x7E, 0x7F, 0xFD, 0xFE, 0xFF))
    assert np.all(np.diff(F.E5M2_TABLE[:0x7C]) > 0)   # positive codes in increasing order


def test_e5m2_round_matches_torch_on_random_values():
    rng = np.random.default_rng(5)
    mag = np.exp2(rng.uniform(-20, 15.8, 200000))
    x = (mag * rng.choice([-1.0, 1.0], mag.size)).astype(np.float32).astype(np.float64)
    x = x[np.abs(x) <= F.E5M2_MAX]
    assert _same_codes(F.e5m2_round(x), _torch_codes(x))


def test_e5m2_round_ties_to_even_at_every_midpoint():
    v = F.E5M2_TABLE[:0x7C]
    mid = (v[:-1] + v[1:]) / 2.0                     # exact in float32 (3 significant bits)
    m32 = mid.astype(np.float32)                      # the float32 neighbours of each midpoint
    x = np.concatenate([mid, -mid, np.nextafter(m32, np.float32(0)).astype(np.float64),
                        np.nextafter(m32, np.float32(np.inf)).astype(np.float64)])
    got = F.e5m2_round(x)
    assert _same_codes(got, _torch_codes(x))
    assert np.all(got[: mid.size] % 2 == 0)          # a tie goes to the even code


def test_e5m2_round_saturates_and_keeps_nan_and_signed_zero():
    got = F.e5m2_round(np.array([57344.0, 61439.0, 1e30, np.inf, -np.inf, -1e30, np.nan, 0.0, -0.0]))
    assert list(got[:6]) == [0x7B, 0x7B, 0x7B, 0x7B, 0xFB, 0xFB]
    assert (got[6] & 0x7C) == 0x7C and (got[6] & 3) != 0
    assert got[7] == 0x00 and got[8] == 0x80


def _torch_recipe(g):
    gt = torch.from_numpy(np.asarray(g, dtype=np.float32))
    amax = gt.abs().amax().to(torch.float32).clamp_min(1e-12)
    step = amax / 57344.0
    return (gt / step).to(torch.float8_e5m2).view(torch.uint8).numpy(), float(step), float(amax)


@pytest.mark.parametrize("std", [1.0, 1e-6, 3e4])
def test_quantize_matches_the_page_recipe_in_torch(std):
    rng = np.random.default_rng(7)
    g = F.bf16_round(rng.standard_normal((300, 257)) * std)
    codes, step, amax = Q.quantize_e5m2(g)
    tcodes, tstep, tamax = _torch_recipe(g)
    assert amax == tamax and step == tstep
    assert _same_codes(codes, tcodes)


def test_quantize_largest_element_lands_on_the_maximum():
    g = F.bf16_round(np.array([[0.5, -3.0, 1.25], [2.0, 0.0, -0.001]]))
    codes, step, amax = Q.quantize_e5m2(g)
    assert amax == 3.0 and step == np.float32(3.0 / 57344.0)
    assert codes[0, 1] == 0xFB and codes[1, 1] == 0x00


def test_quantize_special_cases():
    codes, step, amax = Q.quantize_e5m2(np.zeros((4, 8)))
    assert amax == np.float32(1e-12) and np.all(codes == 0)
    g = np.ones((2, 3))
    g[1, 2] = np.nan
    codes, step, amax = Q.quantize_e5m2(g)
    assert np.isnan(amax) and np.isnan(step)
    assert np.all(((codes & 0x7C) == 0x7C) & ((codes & 3) != 0))


def test_e5m2_dequant_matches_torch_bf16_product():
    rng = np.random.default_rng(9)
    codes = rng.integers(0, 256, size=(3, 40, 64), dtype=np.uint8)
    steps = np.array([1.7e-4, 3.0, 2.0 ** -20], dtype=np.float32)
    got = D.dequant_bits(D.FMT_E5M2_TENSOR, codes, steps, None, 3, 40, 64)
    t = torch.from_numpy(codes).view(torch.float8_e5m2).to(torch.bfloat16)
    ref = t * torch.from_numpy(steps).to(torch.bfloat16).view(3, 1, 1)
    ref_bits = ref.view(torch.int16).numpy().view(np.uint16)
    nan = F.bf16_is_nan_bits(ref_bits)
    assert np.array_equal(F.bf16_is_nan_bits(got), nan)
    assert np.array_equal(got[~nan], ref_bits[~nan])


def test_quantize_then_dequantize_error_is_within_half_a_code_step():
    rng = np.random.default_rng(11)
    g = F.bf16_round(rng.standard_normal((64, 96)))
    codes, step, _ = Q.quantize_e5m2(g)
    back = F.E5M2_TABLE[codes] * step
    # E5M2 keeps 3 significant bits: relative error at most 2^-3 for normal values
    big = np.abs(g) > 2.0 ** -14 * step
    assert np.all(np.abs(back[big] - g[big]) <= np.abs(g[big]) * 2.0 ** -3 + 1e-30)
