"""bsq_dequant on the GPU against the oracle: bit-exact BF16 (every NaN one class)."""

import numpy as np
import pytest
import torch

from block_scaled_gemm_fp8_gb300 import bsq, synth
from tests._util import oracle_deq_bits, same_bits

pytestmark = pytest.mark.gpu

FMTS = [synth.FMT_FP8, synth.FMT_MXFP4, synth.FMT_NVFP4, synth.FMT_FP8_TENSOR, synth.FMT_E5M2_TENSOR]


@pytest.mark.parametrize("fmt", FMTS)
@pytest.mark.parametrize("kind", ["random", "edge", "nan"])
@pytest.mark.parametrize("shape", [(1, 1, 32), (2, 129, 96), (3, 200, 352), (1, 64, 4096)])
def test_dequant_bit_exact(fmt, kind, shape):
    B, R, C = shape
    p = synth.random_codes(fmt, B, R, C, seed=B * 1000 + R + C, scale_kind=kind)
    ref = oracle_deq_bits(p).reshape(B, R, C)
    out = bsq.dequant(p.to("cuda"))
    torch.cuda.synchronize()
    got = synth.bf16_numpy(out).reshape(B, R, C)
    assert same_bits(got, ref), f"mismatches: {(got != ref).sum()}"


@pytest.mark.parametrize("kind", ["random", "edge", "nan"])
@pytest.mark.parametrize("shape", [(2, 3, 48), (1, 5, 16), (3, 7, 80)])
def test_dequant_nvfp4_half_groups(kind, shape):
    """NVFP4 operands whose batch entries hold an odd number of 16-code scale groups (the
    last 4-byte word of a batch entry and the first of the next share a warp load)."""
    B, R, C = shape
    p = synth.random_codes(synth.FMT_NVFP4, B, R, C, seed=7 * B + R + C, scale_kind=kind)
    ref = oracle_deq_bits(p).reshape(B, R, C)
    out = bsq.dequant(p.to("cuda"))
    torch.cuda.synchronize()
    assert same_bits(synth.bf16_numpy(out).reshape(B, R, C), ref)


@pytest.mark.parametrize("fmt", FMTS[:4])   # E5M2 codes come from bsq_quantize_e5m2 (test_gpu_e5m2.py)
def test_dequant_quantized_values(fmt):
    p = synth.make_packed(fmt, 2, 256, 512, 1.0, seed=3, device="cpu")
    ref = oracle_deq_bits(p).reshape(2, 256, 512)
    out = bsq.dequant(p.to("cuda"))
    torch.cuda.synchronize()
    assert same_bits(synth.bf16_numpy(out).reshape(2, 256, 512), ref)


def test_dequant_leaves_no_device_error():
    p = synth.random_codes(synth.FMT_MXFP4, 1, 16, 64, seed=1)
    bsq.dequant(p.to("cuda"))
    st, code = bsq.get_device_error()
    assert st == bsq.BSQ_OK and code == 0
