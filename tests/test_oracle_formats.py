"""Pins for the oracle's code tables and BF16 rounding (CPU only).

Each check compares the oracle with something that is not the oracle: torch's own
E4M3 and BF16 conversions, exact rational arithmetic, the generator's threshold
encoder, or a value the pages state (tests/golden/page_facts.json).
"""

import json
import math
import os
from fractions import Fraction

import numpy as np
import pytest
import torch

from oracle import formats as F

GOLDEN = json.load(open(os.path.join(os.path.dirname(__file__), "golden", "page_facts.json")))


# ------------------------------------------------------------------ E4M3
def test_e4m3_table_matches_torch_float8():
    codes = torch.arange(256, dtype=torch.int32).to(torch.uint8)
    ref = codes.view(torch.float8_e4m3fn).to(torch.float64).numpy()
    tab = F.E4M3_TABLE
    assert np.array_equal(np.isnan(tab), np.isnan(ref))
    fin = ~np.isnan(ref)
    assert np.array_equal(tab[fin], ref[fin])
    assert np.array_equal(np.signbit(tab[fin]), np.signbit(ref[fin]))


def test_e4m3_closed_forms_and_page_max():
    t = F.E4M3_TABLE
    assert t[0x7E] == GOLDEN["e4m3_max"]["value"] == 448.0
    assert np.nanmax(t) == 448.0 and np.nanmin(t) == -448.0
    assert t[0x08] == 2.0 ** -6          # smallest normal
    assert t[0x01] == 2.0 ** -9          # smallest subnormal
    assert t[0x07] == 7 * 2.0 ** -9      # largest subnormal
    assert t[0x38] == 1.0                # exponent field 7 = bias
    assert t[0x00] == 0.0 and not np.signbit(t[0x00])
    assert t[0x80] == 0.0 and np.signbit(t[0x80])
    assert math.isnan(t[0x7F]) and math.isnan(t[0xFF])
    assert np.isnan(t).sum() == 2        # no infinities, two NaNs


def test_e4m3_every_code_round_trips_through_torch_encoder():
    vals = torch.from_numpy(F.E4M3_TABLE.copy())
    back = vals.to(torch.float8_e4m3fn).view(torch.uint8).to(torch.int32).numpy()
    for c in range(256):
        if math.isnan(F.E4M3_TABLE[c]):
            continue
        assert back[c] == c, hex(c)


# ------------------------------------------------------------------ E2M1
def test_e2m1_magnitudes_match_the_pages():
    mags = F.E2M1_TABLE[:8]
    assert list(mags) == GOLDEN["e2m1_magnitudes"]["value"]
    assert len(set(np.abs(F.E2M1_TABLE))) == GOLDEN["e2m1_magnitude_count"]["value"]
    # bit 3 is the sign; codes 8..15 mirror 0..7 (code 8 is -0)
    assert np.array_equal(F.E2M1_TABLE[8:], -F.E2M1_TABLE[:8])
    assert np.signbit(F.E2M1_TABLE[8])


def test_e2m1_every_code_round_trips_through_generator_encoder():
    from block_scaled_gemm_fp8_gb300.synth import e2m1_encode
    codes = e2m1_encode(torch.from_numpy(F.E2M1_TABLE.astype(np.float32))).numpy()
    assert list(codes[:8]) == list(range(8))
    # -0.0 encodes as +0 in the generator (x < 0 is false); every other code round-trips
    assert list(codes[9:]) == list(range(9, 16))


# ------------------------------------------------------------------ E8M0
def test_e8m0_closed_forms():
    t = F.E8M0_TABLE
    assert t[127] == 1.0
    assert t[0] == 2.0 ** -127
    assert t[254] == 2.0 ** 127
    assert t[128] == 2.0 and t[126] == 0.5
    assert math.isnan(t[255])
    for b in range(255):
        assert t[b] == Fraction(2) ** (b - 127)


# ------------------------------------------------------------------ BF16 rounding
def _all_bf16_positive_finite():
    vals = []
    for e in range(255):
        for m in range(128):
            bits = (e << 7) | m
            if e == 0:
                v = Fraction(m, 128) * Fraction(2) ** -126
            else:
                v = (1 + Fraction(m, 128)) * Fraction(2) ** (e - 127)
            vals.append((v, bits))
    return vals


_BF16_POS = None


def _bf16_rne_fraction(x: Fraction):
    """Nearest BF16 to an exact rational by search over all BF16 values; ties to the even pattern."""
    global _BF16_POS
    if _BF16_POS is None:
        _BF16_POS = _all_bf16_positive_finite()
    sign = x < 0
    ax = -x if sign else x
    lo, hi = 0, len(_BF16_POS) - 1
    top = _BF16_POS[-1][0]
    half_ulp_top = Fraction(2) ** 127 * Fraction(1, 256)
    if ax >= top + half_ulp_top:
        return (0xFF80 if sign else 0x7F80)
    while hi - lo > 1:
        mid = (lo + hi) // 2
        if _BF16_POS[mid][0] <= ax:
            lo = mid
        else:
            hi = mid
    a, b = _BF16_POS[lo], _BF16_POS[hi]
    if ax >= b[0]:
        best = b
    else:
        da, db = ax - a[0], b[0] - ax
        best = a if da < db else b if db < da else (a if a[1] % 2 == 0 else b)
    return best[1] | (0x8000 if sign else 0)


def test_bf16_round_matches_torch_on_random_float32_patterns():
    rng = np.random.default_rng(123)
    bits = rng.integers(0, 2 ** 32, size=1_000_000, dtype=np.uint64).astype(np.uint32)
    # extra weight on subnormals, ties (low 16 bits = 0x8000) and the overflow edge
    bits[:50_000] &= 0x807FFFFF
    bits[50_000:100_000] = (bits[50_000:100_000] & 0xFFFF0000) | 0x8000
    bits[100_000:110_000] = 0x7F7F0000 + rng.integers(0, 0x10000, 10_000).astype(np.uint32)
    f32 = bits.view(np.float32)
    keep = ~np.isnan(f32)
    f32 = f32[keep]
    ref = torch.from_numpy(f32.copy()).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    got = F.bf16_bits(F.bf16_round(f32.astype(np.float64)))
    assert np.array_equal(got, ref)


def test_bf16_round_matches_exact_rational_search():
    rng = np.random.default_rng(7)
    xs = []
    pos = _all_bf16_positive_finite()
    for i in rng.integers(0, len(pos) - 1, 600):
        a, b = pos[i][0], pos[i + 1][0]
        xs += [a, (a + b) / 2, a + (b - a) / 3, b - (b - a) / 1000]
    xs += [Fraction(2) ** -133, Fraction(2) ** -134, Fraction(3) * Fraction(2) ** -135,
           Fraction(2) ** 128 - Fraction(2) ** 119, Fraction(2) ** 128 - Fraction(2) ** 120]
    for x in xs:
        for s in (1, -1):
            v = s * x
            got = int(F.bf16_bits(F.bf16_round(np.array([float(v)])))[0])
            if float(v) != v:   # not exactly representable in float64: skip (never happens in the oracle)
                continue
            assert got == _bf16_rne_fraction(v), (v, hex(got))


def test_bf16_round_special_values():
    x = np.array([0.0, -0.0, np.inf, -np.inf, np.nan, 2.0 ** 128, -(2.0 ** 200)])
    r = F.bf16_round(x)
    assert r[0] == 0 and not np.signbit(r[0])
    assert r[1] == 0 and np.signbit(r[1])
    assert r[2] == np.inf and r[3] == -np.inf and np.isnan(r[4])
    assert r[5] == np.inf and r[6] == -np.inf
    assert F.bf16_bits(np.array([np.nan]))[0] == 0x7FC0


def test_fp32_round_matches_numpy_float32_multiply():
    rng = np.random.default_rng(3)
    a = rng.standard_normal(100_000).astype(np.float32)
    b = (rng.standard_normal(100_000) * 1e-3).astype(np.float32)
    exact = a.astype(np.float64) * b.astype(np.float64)   # 48-bit product: exact in float64
    assert np.array_equal(F.fp32_round(exact), (a * b).astype(np.float64))
