"""The quantized-gradient backward (E5M2) against the oracle.

bsq_quantize_e5m2 quantizes a BF16 gradient per tensor with its current amax (AstrAI
fp8.py, `_LinearFp8.backward` in the "hybrid" format): codes, step, amax and the
dequantized copy must equal the oracle's bit for bit (the float32 division and the E5M2
rounding are exact functions of their inputs).  bsq_linear_backward_e5m2 then runs both
products on the dequantized copy; they are held to the GEMM tolerance against the oracle
applied to the oracle's own quantization.
"""

import numpy as np
import pytest
import torch

from block_scaled_gemm_fp8_gb300 import bsq, synth
from oracle import dequant as D
from oracle import formats as F
from oracle import gemm as Gm
from oracle import quantize as Q
from tests._util import assert_gemm, bf16_vals, oracle_deq

pytestmark = pytest.mark.gpu


def _same_codes(a, b):
    nan = lambda c: ((c & 0x7C) == 0x7C) & ((c & 0x03) != 0)
    return np.array_equal(nan(a), nan(b)) and np.array_equal(a[~nan(a)], b[~nan(b)])


def _check_quantize(g_t, margin=0):
    codes, step, amax, deq = bsq.quantize_e5m2(g_t.cuda(), margin=margin)
    torch.cuda.synchronize()
    g = bf16_vals(g_t).reshape(-1)
    rc, rstep, ramax = Q.quantize_e5m2(g, margin)
    got_step, got_amax = float(step.item()), float(amax.item())
    assert (np.isnan(ramax) and np.isnan(got_amax)) or got_amax == ramax, (got_amax, ramax)
    assert (np.isnan(rstep) and np.isnan(got_step)) or got_step == rstep, (got_step, rstep)
    assert _same_codes(codes.cpu().numpy().reshape(-1), rc), "E5M2 codes differ"
    ref_deq = F.bf16_bits(D.dequant_values(D.FMT_E5M2_TENSOR, rc, np.array([rstep], dtype=np.float32), None, 1, 1,
                                           rc.size))
    got = synth.bf16_numpy(deq).reshape(-1)
    nan = F.bf16_is_nan_bits(ref_deq.reshape(-1))
    assert np.array_equal(F.bf16_is_nan_bits(got), nan)
    assert np.array_equal(got[~nan], ref_deq.reshape(-1)[~nan]), "dequantized copy differs"
    assert bsq.get_device_error() == (bsq.BSQ_OK, 0)


@pytest.mark.parametrize("shape", [(1, 8), (3, 7), (300, 257), (1024, 4096)])
@pytest.mark.parametrize("std", [1.0, 1e-30, 3e4])
def test_quantize_bit_exact(shape, std):
    _check_quantize(synth.randn(shape, std, shape[0] + shape[1], "cpu", torch.bfloat16))


@pytest.mark.parametrize("margin", [0, 3, 30])
def test_quantize_margin_saturates(margin):
    _check_quantize(synth.randn((64, 96), 1.0, 3, "cpu", torch.bfloat16), margin)


def test_quantize_special_values():
    z = torch.zeros((16, 24), dtype=torch.bfloat16)
    _check_quantize(z)                                  # amax at its 1e-12 floor, every code 0
    g = synth.randn((16, 24), 1.0, 4, "cpu", torch.bfloat16)
    g[3, 5] = float("nan")
    _check_quantize(g)                                  # NaN amax: every code NaN
    g = synth.randn((16, 24), 1.0, 5, "cpu", torch.bfloat16)
    g[7, 1] = float("-inf")
    _check_quantize(g)                                  # infinite step: finite -> 0, inf / inf -> NaN
    _check_quantize(torch.zeros((0,), dtype=torch.bfloat16))


def test_quantize_every_bf16_pattern():
    """All 65536 BF16 bit patterns (NaNs included) in one tensor, then without NaN and inf."""
    bits = torch.arange(65536, dtype=torch.int32).to(torch.int16).view(torch.bfloat16)
    _check_quantize(bits.clone())
    finite = bits[torch.isfinite(bits.float())]
    _check_quantize(finite.clone())


def test_quantize_bit_exact_across_steps():
    """Every finite BF16 value of magnitude up to amax, for 48 amax values from 2^-30 to
    2^30 and margins 0..3: the kernel divides through the reciprocal of the step and takes
    the IEEE division where the product lies within a few ulps of an E5M2 rounding
    midpoint or below 2^-13; every element must still match the float32 quotient's code."""
    bits = torch.arange(65536, dtype=torch.int32).to(torch.int16).view(torch.bfloat16)
    finite = bits[torch.isfinite(bits.float())]
    rng = np.random.default_rng(17)
    for a in rng.uniform(-30.0, 30.0, 48):
        amax = torch.tensor([2.0 ** a * rng.uniform(1.0, 2.0)]).to(torch.bfloat16)
        g = torch.cat([finite[finite.float().abs() <= amax.float()], amax, -amax])
        _check_quantize(g.clone(), margin=int(rng.integers(0, 4)))


@pytest.mark.parametrize("fmt", [synth.FMT_MXFP4, synth.FMT_FP8])
@pytest.mark.parametrize("M,N,K", [(300, 256, 384), (8, 512, 256), (1024, 1024, 1024)])
@pytest.mark.parametrize("needs", [3, 1, 2])
def test_linear_backward_e5m2(fmt, M, N, K, needs):
    W = synth.make_packed(fmt, 1, N, K, 0.5, seed=M + N, device="cpu")
    X = synth.make_packed(fmt, 1, M, K, 1.0, seed=M + K, device="cpu")
    G = synth.randn((M, N), 1e-2, M + N + K, "cpu", torch.bfloat16)
    gx, gw, step, amax = bsq.linear_backward_e5m2(G.cuda(), W.to("cuda"), X.to("cuda"), needs=needs)
    torch.cuda.synchronize()
    codes, rstep, ramax = Q.quantize_e5m2(bf16_vals(G))
    assert float(step.item()) == rstep and float(amax.item()) == ramax
    gq = D.dequant_values(D.FMT_E5M2_TENSOR, codes.reshape(1, M, N), np.array([rstep], dtype=np.float32), None,
                          1, M, N)[0]
    w, x = oracle_deq(W)[0], oracle_deq(X)[0]
    if needs & 1:
        assert_gemm(bf16_vals(gx), Gm.dgrad(gq, w), gq, w, N, f"e5m2 dgrad fmt={fmt}")
    else:
        assert gx is None
    if needs & 2:
        assert_gemm(bf16_vals(gw), Gm.wgrad(gq, x), gq, x, M, f"e5m2 wgrad fmt={fmt}")
    else:
        assert gw is None
    assert bsq.get_device_error() == (bsq.BSQ_OK, 0)
